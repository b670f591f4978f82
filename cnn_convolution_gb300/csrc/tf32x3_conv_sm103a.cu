// Split-precision tensor-core convolution for fp32 tensors on sm_103a (3xTF32).
//
// The fp32 path of "Enabling Memory-efficient Im2win Convolution with
// Multi-precision Support on GPU CUDA and Tensor Cores" (abstract: the same
// convolution across precisions) moved from CUDA cores to tensor cores while
// keeping fp32 accuracy.  Blackwell has no full-rate fp32 MMA, but it has
// TF32 (fp32 range, 11 significant bits).  Every fp32 operand a is split, as
// it is staged into shared memory, into
//     a_hi = tf32_rn(a),   a_lo = tf32_rn(a - a_hi)       (a - a_hi is exact)
// and each product is formed as x_hi*w_hi + x_hi*w_lo + x_lo*w_hi: three
// kind::tf32 MMAs into one fp32 accumulator in tensor memory.  What is left
// out per product -- x_lo*w_lo and the two split residues |a - a_hi - a_lo|
// <= 2^-22 |a| -- is at most about 3 * 2^-22 |x||w|, i.e. below 7.2e-7 of
// sum |x||w| over a whole output even if every term erred the same way.
//
// GEMM view as in "GPU-Accelerating MSCRED with CUDA, im2col, GEMM, and a
// Custom PyTorch Extension" (section "Transforming Conv2D into im2col and
// GEMM"), without materialising the im2col matrix: D[m, k] = sum_g
// A[m, g] * W[k, g] with m = (n, p, q) and g the reduction index in the
// weight tensor's own order -- (c, r, s) for KCRS weights (NCHW), (r, s, c)
// for KRSC weights (NHWC) -- so every weight row is contiguous.  A[m, g] is
// gathered from x through a per-CTA table g -> (offset, r*dil, s*dil), zero
// outside the image, exactly like the CUDA-core kernel's tap table.
//
// Warp roles: warps 0..3 epilogue (warp w owns accumulator lanes 32w..32w+31),
// warps 4..3+NPROD gather + split + store the A and B tiles of each stage in
// the 128-byte-swizzled K-major layout the MMA descriptors expect, the last
// warp allocates tensor memory and issues the MMAs.  A stage covers 32
// reduction elements (one 128-byte row of fp32); tiles are 128 output pixels
// x BN output channels; the accumulator is double-buffered in tensor memory
// so the epilogue of one tile overlaps the main loop of the next; CTAs are
// persistent.  Every mbarrier wait is bounded (see ptx_sm103a.cuh).

#include <cuda.h>

#include <algorithm>
#include <atomic>
#include <cstdint>

#include "internal.h"
#include "ptx_sm103a.cuh"

namespace conv2d {
namespace {

using namespace sm103a;

constexpr int kTfBM = 128;                    // output pixels per tile (MMA M, TMEM lanes)
constexpr int kTfBK = 32;                     // reduction elements per stage (128 B of fp32)
constexpr int kTfATile = kTfBM * kTfBK * 4;   // one A operand tile: 16 KB

// D(tmem) (+)= A(smem) * B(smem)^T, M=128, N from idesc, K=8 (TF32).
__device__ __forceinline__ void mma_tf32(uint32_t d_tmem, uint64_t a_desc, uint64_t b_desc,
                                         uint32_t idesc, uint32_t accumulate) {
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "setp.ne.b32 p, %4, 0;\n\t"
        "tcgen05.mma.cta_group::1.kind::tf32 [%0], %1, %2, %3, p;\n\t}" ::"r"(d_tmem),
        "l"(a_desc), "l"(b_desc), "r"(idesc), "r"(accumulate)
        : "memory");
}

// D(tmem) (+)= A(tmem) * B(smem)^T: A is 128 lanes x 8 columns of TF32 values
// (lane = row, column = reduction element) starting at a_tmem.
__device__ __forceinline__ void mma_tf32_ts(uint32_t d_tmem, uint32_t a_tmem, uint64_t b_desc,
                                            uint32_t idesc, uint32_t accumulate) {
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "setp.ne.b32 p, %4, 0;\n\t"
        "tcgen05.mma.cta_group::1.kind::tf32 [%0], [%1], %2, %3, p;\n\t}" ::"r"(d_tmem),
        "r"(a_tmem), "l"(b_desc), "r"(idesc), "r"(accumulate)
        : "memory");
}

// Instruction descriptor, kind::tf32: fp32 accumulate, A and B TF32, both K-major.
__host__ __device__ constexpr uint32_t make_idesc_tf32(int n) {
    return (1u << 4)                                   // D format: f32
           | (2u << 7)                                 // A format: TF32
           | (2u << 10)                                // B format: TF32
           | ((uint32_t)(n >> 3) << 17)                // N / 8
           | ((uint32_t)(kTfBM >> 4) << 24);           // M / 16
}

// fp32 -> nearest TF32 value (ties away from zero), on the bit pattern:
// adding half a TF32 unit (bit 12) to the sign-magnitude encoding and
// clearing the 13 low mantissa bits rounds the magnitude; a carry moves into
// the exponent as it should.  Integer ALU work at full rate, unlike a
// conversion instruction.
__device__ __forceinline__ uint32_t tf32_rn(float a) {
    return (__float_as_uint(a) + 0x1000u) & 0xFFFFE000u;
}

// Split four values into their TF32 high and low parts.
__device__ __forceinline__ void split4(const float (&v)[4], uint32_t (&hi)[4], uint32_t (&lo)[4]) {
#pragma unroll
    for (int e = 0; e < 4; ++e) {
        hi[e] = tf32_rn(v[e]);
        lo[e] = tf32_rn(v[e] - __uint_as_float(hi[e]));
    }
}

// Optional timeline trace of CTA 0 (compile with -DCONV2D_TC_TRACE; off in
// the library build), read back with conv2d_tf_trace_dump().
#ifdef CONV2D_TC_TRACE
__device__ unsigned long long g_tf_trace[4][8192];
__device__ unsigned int g_tf_trace_n[4];
// one tracing thread per role keeps its own event count in a register
#define TF_TRACE(role, tag)                                                                  \
    do {                                                                                     \
        if (blockIdx.x == 0) {                                                               \
            if (tr_n < 8192u)                                                                \
                g_tf_trace[role][tr_n] =                                                     \
                    ((unsigned long long)(tag) << 48) | ((unsigned long long)clock64() & 0xFFFFFFFFFFFFull); \
            ++tr_n;                                                                          \
            g_tf_trace_n[role] = tr_n;                                                       \
        }                                                                                    \
    } while (0)
#else
#define TF_TRACE(role, tag) \
    do {                    \
    } while (0)
#endif

struct TfParams {
    const float *x;
    const float *w;
    const float *bias;
    float *y;
    unsigned int *status;
    int64_t M;          // N*P*Q
    int64_t img;        // elements of x per image (C*H*W)
    int K, Kg, KT;      // output channels, reduction length, stages per tile
    int C, H, W, S, RS;
    int Q, PQ;
    int stride, pad, dil;
    int n_tiles_n, total_tiles;
    int nhwc;
    int rs_mask;        // R*S <= 63: taps carry their (r, s) index, tested against a per-tile mask
    int R;
    // NCHW 2x2 filter: reduction index g = 4c + 2r + s, so a 4-element chunk is
    // one input channel's four taps and offsets follow from g without the table
    int tap4, HW, dilW;
    int w_vec;          // Kg % 4 == 0 and w 16-byte aligned: weight rows load as float4
    int y_vec;          // NHWC, K % 4 == 0 and y 16-byte aligned: outputs store as float4
    // ConvLSTM cell epilogue (LSTM instantiations only): K = 4*Ch gate columns,
    // read from gate-major weight rows in interleaved order (column 4u+gate is
    // weight row gate*Ch + u), so that each group of 4 columns holds the
    // i, f, o, g pre-activations of hidden unit u
    // transposed-convolution residue class (dv = 1): the GEMM pixels are the
    // outputs (a + st*i, b + st*j) of y [N][K][dv_H][dv_W]; the reduction index
    // g = (k_in, rj, sl) takes filter tap (dv_r[rj], dv_s[sl]) of w [K_in][K][R][S]
    // and input pixel (i + dv_e[rj], j + dv_f[sl]) of x [N][K_in][H][W]
    int dv, dv_H, dv_W, dv_a, dv_b, dv_st, dv_J, dv_L, dv_R, dv_S;
    int dv_e[8], dv_f[8], dv_r[8], dv_s[8];
    int lstm_ch;
    const float *c_prev;   // [N][Ch][P][Q]
    float *c_next;         // [N][Ch][P][Q]
    float *h_next;         // image n at h_next + n * h_img, [Ch][P][Q] inside
    int64_t h_img;
};

__device__ __forceinline__ float sigmoidf_(float z) { return 1.0f / (1.0f + expf(-z)); }

// Tensor memory: columns [0, 2 BN) hold the correction accumulators (x_hi*w_lo
// + x_lo*w_hi) of two tiles in flight; NSLOT slots of BN columns after them
// receive the x_hi*w_hi partial sum of one 32-element stage each.  With the
// A operand in tensor memory (AT), STAGES stages of 64 columns follow: the
// stage's 32 A_hi columns, then its 32 A_lo columns (lane = output pixel).
template <int BN, bool AT = false, int STAGES = 1>
struct TfTmem {
    static constexpr int kACols = AT ? 64 * STAGES : 0;
    static constexpr int kFree = (512 - 2 * BN - kACols) / BN;
    static constexpr int kSlots = AT ? (kFree > 6 ? 6 : kFree) : (BN >= 128 ? 2 : 6);
    static constexpr int kACol0 = 2 * BN + kSlots * BN;
    static constexpr int kUsed = kACol0 + kACols;
    static constexpr uint32_t kCols = kUsed <= 32 ? 32 : kUsed <= 64 ? 64 : kUsed <= 128 ? 128
                                      : kUsed <= 256 ? 256 : 512;
    static_assert(kSlots >= 2 && kUsed <= 512, "tensor memory");
};

// Shared memory: STAGES x ([A_hi, A_lo unless AT][, B_hi, B_lo]), barriers, then -- with
// resident weights (RESB) -- the split weights of every stage of the CTA's
// output-channel tile (KT x (B_hi, B_lo)), then the tap table.
template <int BN, int STAGES, bool RESB = false, bool AT = false>
struct TfSmem {
    static constexpr int kBTile = BN * kTfBK * 4;
    static constexpr int kStage = (AT ? 0 : 2 * kTfATile) + (RESB ? 0 : 2 * kBTile);
    static constexpr int kSlots = TfTmem<BN, AT, STAGES>::kSlots;
    static constexpr size_t kBarOffset = (size_t)STAGES * kStage;
    // full[S], empty[S], slot_full[NS], slot_empty[NS], corr_full[2], corr_empty[2], drain,
    // weights-ready; then the tensor-memory address and the abort flag
    static constexpr size_t kBarBytes = (2 * STAGES + 2 * kSlots + 6) * 8;
    static constexpr size_t kResBOffset = (kBarOffset + kBarBytes + 16 + 1023) / 1024 * 1024;
    static constexpr size_t tap_offset(int kt) {
        return RESB ? kResBOffset + (size_t)kt * 2 * kBTile : (kBarOffset + kBarBytes + 16 + 15) / 16 * 16;
    }
    // tap table (8 bytes per reduction index), then the weight-offset table of
    // transposed convolutions (4 bytes per index)
    static constexpr size_t bytes(int kt) { return tap_offset(kt) + (size_t)kt * kTfBK * 12 + 1024; }
};

template <int BN> constexpr int tf_epi_warps() { return BN >= 64 ? 8 : 4; }
template <int BN, int NPROD> constexpr int tf_threads() { return 32 * (tf_epi_warps<BN>() + NPROD + 1); }

// Accuracy: the tensor cores add each MMA's products into the fp32
// accumulator with their own (not round-to-nearest) alignment and rounding,
// so one long accumulation chain loses bits in proportion to its length.
// Hence the x_hi*w_hi term -- the only one of full magnitude -- is summed in
// tensor memory over one stage only (4 MMAs of K=8) and the stage sums are
// added in fp32 registers by the epilogue warps; the correction terms, 2^-11
// smaller, stay in one accumulator per tile.
//
// Producer groups: the NPROD producer warps form NGRP groups, and stage f of
// the CTA's sequence is filled by group f % NGRP alone.  A producer warp's
// pass over a stage is a chain of latencies (tap reads feeding the load
// addresses, the wait for the stage to be free, the stores, the proxy fence
// and the arrival) that more warps on the same stage do not shorten; with
// two groups, two stages are filled at once and each warp pays the chain
// once per two stages for twice the elements.  With one group a warp issues
// the loads of its next stage before storing the current one; with several,
// it issues its loads and then waits for the stage to be free, so that wait
// overlaps the loads' latency.
// AT: the A operand lives in tensor memory.  The producers write each stage's
// A_hi / A_lo columns with tcgen05.st (lane = their output pixel) and the
// MMAs read A from there, so shared memory carries only the weights: the
// tensor cores' operand reads no longer compete with the producers' stores.
template <int BN, int STAGES, int NPROD, bool LSTM, bool RESB, int NGRP, bool AT>
__global__ void __launch_bounds__(tf_threads<BN, NPROD>(), 1) tf32x3_conv_kernel(const TfParams p) {
    using L = TfSmem<BN, STAGES, RESB, AT>;
    using TM = TfTmem<BN, AT, STAGES>;
    constexpr uint32_t kIdesc = make_idesc_tf32(BN);
    constexpr int kSlots = TM::kSlots;
    constexpr int kEpiWarps = tf_epi_warps<BN>();
    constexpr int kEpiThreads = 32 * kEpiWarps;
    static_assert(NPROD <= 32 && kEpiWarps <= 32, "arrival counts");
    constexpr int kCpt = BN * 4 / kEpiWarps;                     // accumulator columns per epilogue thread
    constexpr int kProd = 32 * NPROD;                            // producer threads
    constexpr int kMmaWarp = kEpiWarps + NPROD;
    static_assert(NGRP >= 1 && NPROD % NGRP == 0, "producer groups");
    constexpr int kGrpWarps = NPROD / NGRP;                      // producer warps per group
    constexpr int kGrpThr = 32 * kGrpWarps;
    constexpr int kChunks = 8 * kTfBM / kGrpThr;                 // A chunks (4 values) per thread per stage
    constexpr int kBIter = BN * 8 / kGrpThr;                     // B chunks per thread per stage
    static_assert(kChunks >= 1 && kChunks * kGrpThr == 8 * kTfBM, "producer split (A)");
    static_assert(RESB || (kBIter >= 1 && kBIter * kGrpThr == 8 * BN), "producer split (B)");
    static_assert(kCpt % 16 == 0, "epilogue columns");

    extern __shared__ uint8_t smem_raw[];
    // 1024-byte aligned base, derived from the shared array itself so that
    // the compiler keeps the shared address space (plain shared loads)
    uint8_t *smem = smem_raw + ((1024u - (smem_u32(smem_raw) & 1023u)) & 1023u);
    const uint32_t smem_base = smem_u32(smem);
    const uint32_t bar_base = smem_base + (uint32_t)L::kBarOffset;
    auto full_bar = [&](int s) { return bar_base + 8u * s; };
    auto empty_bar = [&](int s) { return bar_base + 8u * (STAGES + s); };
    auto slotf_bar = [&](int s) { return bar_base + 8u * (2 * STAGES + s); };
    auto slote_bar = [&](int s) { return bar_base + 8u * (2 * STAGES + kSlots + s); };
    auto corrf_bar = [&](int a) { return bar_base + 8u * (2 * STAGES + 2 * kSlots + a); };
    auto corre_bar = [&](int a) { return bar_base + 8u * (2 * STAGES + 2 * kSlots + 2 + a); };
    const uint32_t drain_bar = bar_base + 8u * (2 * STAGES + 2 * kSlots + 4);
    const uint32_t bres_bar = bar_base + 8u * (2 * STAGES + 2 * kSlots + 5);
    uint32_t *tmem_holder = reinterpret_cast<uint32_t *>(smem + L::kBarOffset + L::kBarBytes);
    volatile int *abort_flag = reinterpret_cast<volatile int *>(smem + L::kBarOffset + L::kBarBytes + 4);
    int2 *taps = reinterpret_cast<int2 *>(smem + L::tap_offset(p.KT));
    int *wtaps = reinterpret_cast<int *>(taps + p.KT * kTfBK);     // transposed convolution only

    const int warp = threadIdx.x / 32;
    const int lane = threadIdx.x % 32;
#ifdef CONV2D_TC_TRACE
    unsigned tr_n = 0;
#endif

    // Tap table: reduction index g -> (offset of x[g] from the output pixel's
    // input origin, tap id).  With R*S <= 63 the tap id is r*S + s, looked up
    // in a per-tile bitmask of the taps that fall inside the image; entries
    // past Kg use id 63, never set.  Otherwise it is (r*dil) << 16 | s*dil and
    // entries past Kg carry a row offset of -32768, which no pixel reaches.
    for (int g = threadIdx.x; g < p.KT * kTfBK; g += blockDim.x) {
        int2 t;
        if (p.dv) {
            // transposed convolution: g = (k_in, rj, sl); offsets may be negative
            int wo = 0;
            t.x = 0;
            t.y = (int)0x80000000u;
            if (g < p.Kg) {
                const int JL = p.dv_J * p.dv_L;
                const int k = g / JL, rs = g - k * JL;
                const int rj = rs / p.dv_L, sl = rs - rj * p.dv_L;
                const int dh = p.dv_e[rj], dw = p.dv_f[sl];
                t.x = (k * p.H + dh) * p.W + dw;
                t.y = (dh << 16) | (dw & 0xFFFF);
                wo = (k * p.K * p.dv_R + p.dv_r[rj]) * p.dv_S + p.dv_s[sl];
            }
            taps[g] = t;
            wtaps[g] = wo;
            continue;
        }
        if (g < p.Kg) {
            int c, rs;
            if (p.nhwc) {
                rs = g / p.C;
                c = g - rs * p.C;
            } else {
                c = g / p.RS;
                rs = g - c * p.RS;
            }
            const int r = rs / p.S, s = rs - r * p.S;
            const int dh = r * p.dil, dw = s * p.dil;
            t.x = p.nhwc ? (dh * p.W + dw) * p.C + c : (c * p.H + dh) * p.W + dw;
            t.y = p.rs_mask ? rs : (dh << 16) | dw;
        } else {
            t.x = 0;
            t.y = p.rs_mask ? 63 : (int)0x80000000u;
        }
        taps[g] = t;
    }
    if (threadIdx.x == 0) {
        for (int s = 0; s < STAGES; ++s) {
            mbar_init(full_bar(s), kGrpWarps);      // one arrival per warp of the filling group
            mbar_init(empty_bar(s), 1);
        }
        for (int s = 0; s < kSlots; ++s) {
            mbar_init(slotf_bar(s), 1);
            mbar_init(slote_bar(s), kEpiWarps);     // one arrival per epilogue warp
        }
        for (int a = 0; a < 2; ++a) {
            mbar_init(corrf_bar(a), 1);
            mbar_init(corre_bar(a), kEpiWarps);
        }
        mbar_init(drain_bar, 1);
        mbar_init(bres_bar, NPROD);
        *abort_flag = 0;
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
        asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
    }
    if (warp == kMmaWarp) {
        tmem_alloc(smem_u32(tmem_holder), TM::kCols);
        tmem_relinquish();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem_base = *tmem_holder;
    // everything above depends on parameters only; x, w, bias, c and y are
    // touched after the previous kernel on the stream has finished
    pdl_launch_dependents();
    pdl_wait();
    auto a_hi = [&](int s) { return smem_base + (uint32_t)(s * L::kStage); };
    auto a_lo = [&](int s) { return smem_base + (uint32_t)(s * L::kStage + kTfATile); };
    // weight tiles of stage s (streamed) or of reduction stage ks (resident)
    auto b_hi = [&](int s) {
        return RESB ? smem_base + (uint32_t)(L::kResBOffset + (size_t)s * 2 * L::kBTile)
                    : smem_base + (uint32_t)(s * L::kStage + (AT ? 0 : 2 * kTfATile));
    };
    auto b_lo = [&](int s) { return b_hi(s) + (uint32_t)L::kBTile; };

    if (warp >= kEpiWarps && warp < kMmaWarp) {
        // ---------------------------------------------------------- producers
        // The CTA's (tile, stage) pairs are numbered f = 0, 1, ...; group grp
        // fills f = grp, grp + NGRP, ...  Thread gpt of a group owns A row
        // (gpt % 128) and kChunks of its 8 16-byte chunks; B rows are shared
        // out 8 chunks per row across the group's threads.  Stores follow the
        // 128-byte swizzle: chunk j of row r sits at position j ^ (r % 8).
        const int pt = threadIdx.x - kEpiThreads;
        const int grp = pt / kGrpThr;
        const int gpt = pt - grp * kGrpThr;
        const int row = gpt & (kTfBM - 1);
        const int chunk0 = (gpt / kTfBM) * kChunks;
        const uint32_t a_row_off = (uint32_t)row * 128u;
        const uint32_t row_sw = (uint32_t)(row & 7);
        const int my_tiles = (p.total_tiles - (int)blockIdx.x + (int)gridDim.x - 1) / (int)gridDim.x;
        const int nf = my_tiles * p.KT;
        // loader position (tile, stage) and the row state of that tile
        int l_tile = (int)blockIdx.x, l_ks = grp, cur_tile = -1;
        while (l_ks >= p.KT) { l_ks -= p.KT; l_tile += (int)gridDim.x; }
        int h0 = -65536, w0 = 0, base = 0, k0 = 0;
        uint64_t vmask = 0;          // bit r*S+s: tap (r, s) of this row's pixel lies inside the image
        const float *ximg = p.x;
        const int4 *taps4 = reinterpret_cast<const int4 *>(taps);   // two taps per 16 bytes
        bool ok = true;

        auto load = [&](float (&va)[kChunks][4], float (&vb)[kBIter][4]) {
            if (pt == 0) TF_TRACE(0, 1);
            const int ks = l_ks;
            if (l_tile != cur_tile) {
                cur_tile = l_tile;
                const int tm = l_tile / p.n_tiles_n;
                k0 = (l_tile - tm * p.n_tiles_n) * BN;
                const int64_t m = (int64_t)tm * kTfBM + row;
                h0 = -65536;
                w0 = 0;
                base = 0;
                ximg = p.x;
                if (m < p.M) {
                    const int n = (int)(m / p.PQ);
                    const int pq = (int)(m - (int64_t)n * p.PQ);
                    const int pp = pq / p.Q, q = pq - pp * p.Q;
                    h0 = pp * p.stride - p.pad;
                    w0 = q * p.stride - p.pad;
                    ximg = p.x + (int64_t)n * p.img;
                    base = p.nhwc ? (h0 * p.W + w0) * p.C : h0 * p.W + w0;
                }
                if (p.rs_mask) {
                    vmask = 0;
                    if (m < p.M) {
                        uint32_t wbits = 0;
                        for (int s = 0; s < p.S; ++s)
                            wbits |= ((unsigned)(w0 + s * p.dil) < (unsigned)p.W ? 1u : 0u) << s;
                        for (int r = 0; r < p.R; ++r)
                            if ((unsigned)(h0 + r * p.dil) < (unsigned)p.H)
                                vmask |= (uint64_t)wbits << (r * p.S);
                    }
                }
            }
            l_ks += NGRP;
            while (l_ks >= p.KT) { l_ks -= p.KT; l_tile += (int)gridDim.x; }
            const float *xrow = ximg + base;   // the pixel's input origin (may lie in the padding)
            if (p.tap4) {
                // chunk j is input channel ks*8 + chunk0 + j; element e is tap
                // (e >> 1, e & 1), bit e of the tile's tap mask
                const int cb = ks * (kTfBK / 4) + chunk0;
#pragma unroll
                for (int j = 0; j < kChunks; ++j) {
                    const bool cin = cb + j < p.C;
                    const int coff = cin ? (cb + j) * p.HW : 0;
#pragma unroll
                    for (int e = 0; e < 4; ++e)
                        va[j][e] = ldg_or_zero(xrow + coff + (e >> 1) * p.dilW + (e & 1) * p.dil,
                                               cin && ((vmask >> e) & 1u));
                }
            } else if (p.rs_mask) {
                // all taps of this thread's chunks first (shared broadcast
                // reads), then all the global loads
                int4 tv[kChunks * 2];
#pragma unroll
                for (int q = 0; q < kChunks * 2; ++q) tv[q] = taps4[(ks * kTfBK + chunk0 * 4) / 2 + q];
#pragma unroll
                for (int j = 0; j < kChunks; ++j) {
#pragma unroll
                    for (int e = 0; e < 4; ++e) {
                        const int4 t2 = tv[j * 2 + (e >> 1)];
                        const int off = (e & 1) ? t2.z : t2.x;
                        const int rs = (e & 1) ? t2.w : t2.y;
                        va[j][e] = ldg_or_zero(xrow + off, (vmask >> rs) & 1u);
                    }
                }
            } else {
                int4 tv[kChunks * 2];
#pragma unroll
                for (int q = 0; q < kChunks * 2; ++q) tv[q] = taps4[(ks * kTfBK + chunk0 * 4) / 2 + q];
#pragma unroll
                for (int j = 0; j < kChunks; ++j) {
#pragma unroll
                    for (int e = 0; e < 4; ++e) {
                        const int4 t2 = tv[j * 2 + (e >> 1)];
                        const int off = (e & 1) ? t2.z : t2.x;
                        const int hw = (e & 1) ? t2.w : t2.y;
                        const int dh = hw >> 16, dw = (int)(short)(hw & 0xFFFF);
                        const bool in = (unsigned)(h0 + dh) < (unsigned)p.H &&
                                        (unsigned)(w0 + dw) < (unsigned)p.W;
                        va[j][e] = ldg_or_zero(xrow + off, in);
                    }
                }
            }
#pragma unroll
            for (int it = 0; it < (RESB ? 0 : kBIter); ++it) {
                const int i = gpt + it * kGrpThr;
                const int k = k0 + (i >> 3);
                const int g = ks * kTfBK + (i & 7) * 4;
                const int wrow = LSTM ? (k & 3) * p.lstm_ch + (k >> 2) : k;
                const float *wr = p.w + (int64_t)wrow * p.Kg + g;
                if (p.dv) {
                    // w [K_in][K][R][S]: element (k, g) at wtaps[g] + k*R*S
#pragma unroll
                    for (int e = 0; e < 4; ++e) {
                        const bool in = k < p.K && g + e < p.Kg;
                        vb[it][e] = ldg_or_zero(p.w + (in ? wtaps[g + e] + k * p.dv_R * p.dv_S : 0), in);
                    }
                } else if (p.w_vec) {
                    ldg4_or_zero(wr, k < p.K && g < p.Kg, vb[it]);
                } else {
#pragma unroll
                    for (int e = 0; e < 4; ++e) vb[it][e] = ldg_or_zero(wr + e, k < p.K && g + e < p.Kg);
                }
            }
        };
        auto store = [&](int f, const float (&va)[kChunks][4], const float (&vb)[kBIter][4]) -> bool {
            if (pt == 0) TF_TRACE(0, 6);
            const int stage = f % STAGES;
            const uint32_t phase = (uint32_t)(f / STAGES) & 1u;
            // every lane observes the MMAs' release of the stage itself before
            // overwriting it (measured faster on the encoder layers than one
            // waiting lane and a warp shuffle)
            if (!__all_sync(0xffffffffu, mbar_wait(empty_bar(stage), phase ^ 1u, abort_flag, p.status)))
                return false;
            if (pt == 0) TF_TRACE(0, 2);
            if constexpr (AT) {
                // this warp's 32 lanes are its pixels' accumulator rows; the
                // thread writes its kChunks * 4 reduction elements of the
                // stage into the A_hi and A_lo columns
                tc_fence_after();
                // in pieces of at most 4 chunks (16 columns), to bound registers
                constexpr int kPc = kChunks < 4 ? kChunks : 4;
                const uint32_t ta = tmem_base + ((uint32_t)((warp & 3) * 32) << 16) +
                                    (uint32_t)(TM::kACol0 + stage * 64 + chunk0 * 4);
#pragma unroll
                for (int j0 = 0; j0 < kChunks; j0 += kPc) {
                    uint32_t hi[kPc * 4], lo[kPc * 4];
#pragma unroll
                    for (int j = 0; j < kPc; ++j) {
                        uint32_t h4[4], l4[4];
                        split4(va[j0 + j], h4, l4);
#pragma unroll
                        for (int e = 0; e < 4; ++e) {
                            hi[4 * j + e] = h4[e];
                            lo[4 * j + e] = l4[e];
                        }
                    }
                    tmem_st<kPc * 4>(ta + (uint32_t)(j0 * 4), hi);
                    tmem_st<kPc * 4>(ta + 32u + (uint32_t)(j0 * 4), lo);
                }
                tmem_st_wait();
            } else {
#pragma unroll
                for (int j = 0; j < kChunks; ++j) {
                    uint32_t hi[4], lo[4];
                    split4(va[j], hi, lo);
                    const uint32_t off = a_row_off + ((((uint32_t)(chunk0 + j)) ^ row_sw) << 4);
                    st_shared_v4(a_hi(stage) + off, hi[0], hi[1], hi[2], hi[3]);
                    st_shared_v4(a_lo(stage) + off, lo[0], lo[1], lo[2], lo[3]);
                }
            }
#pragma unroll
            for (int it = 0; it < (RESB ? 0 : kBIter); ++it) {
                const int i = gpt + it * kGrpThr;
                const int kr = i >> 3, cj = i & 7;
                uint32_t hi[4], lo[4];
                split4(vb[it], hi, lo);
                const uint32_t off = (uint32_t)kr * 128u + ((((uint32_t)cj) ^ (uint32_t)(kr & 7)) << 4);
                st_shared_v4(b_hi(stage) + off, hi[0], hi[1], hi[2], hi[3]);
                st_shared_v4(b_lo(stage) + off, lo[0], lo[1], lo[2], lo[3]);
            }
            // make this thread's generic-proxy stores visible to the tensor cores
            if (pt == 0) TF_TRACE(0, 5);
            // each thread makes its generic-proxy stores (and, with AT, its
            // completed tensor-memory stores) visible to the tensor cores;
            // then one lane per warp arrives for the whole warp
            fence_proxy_async_smem();
            if (AT) tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(full_bar(stage));
            if (pt == 0) TF_TRACE(0, 3);
            return true;
        };

        if (RESB && nf > 0) {
            // Split every stage's weights of this CTA's output-channel tile
            // once (the tile is the same for all the CTA's tiles: the launch
            // keeps gridDim a multiple of the tile count along K).
            const int tn = (int)blockIdx.x % p.n_tiles_n;
            const int kw0 = tn * BN;
            const int total = p.KT * BN * 8;
            for (int i0 = pt; i0 < total; i0 += kProd * 4) {
                float vw[4][4];
#pragma unroll
                for (int u = 0; u < 4; ++u) {
                    const int i = i0 + u * kProd;
                    const int ks = i / (BN * 8), r8 = i - ks * (BN * 8);
                    const int k = kw0 + (r8 >> 3);
                    const int g = ks * kTfBK + (r8 & 7) * 4;
                    const int wrow = LSTM ? (k & 3) * p.lstm_ch + (k >> 2) : k;
                    const bool rowin = i < total && k < p.K;
                    const float *wr = p.w + (rowin ? (int64_t)wrow * p.Kg + g : 0);
                    if (p.dv) {
#pragma unroll
                        for (int e = 0; e < 4; ++e) {
                            const bool in = rowin && g + e < p.Kg;
                            vw[u][e] = ldg_or_zero(p.w + (in ? wtaps[g + e] + k * p.dv_R * p.dv_S : 0), in);
                        }
                    } else if (p.w_vec) {
                        ldg4_or_zero(wr, rowin && g < p.Kg, vw[u]);
                    } else {
#pragma unroll
                        for (int e = 0; e < 4; ++e) vw[u][e] = ldg_or_zero(wr + e, rowin && g + e < p.Kg);
                    }
                }
#pragma unroll
                for (int u = 0; u < 4; ++u) {
                    const int i = i0 + u * kProd;
                    if (i >= total) break;
                    const int ks = i / (BN * 8), r8 = i - ks * (BN * 8);
                    const int kr = r8 >> 3, cj = r8 & 7;
                    uint32_t hi[4], lo[4];
                    split4(vw[u], hi, lo);
                    const uint32_t off = (uint32_t)kr * 128u + ((((uint32_t)cj) ^ (uint32_t)(kr & 7)) << 4);
                    st_shared_v4(b_hi(ks) + off, hi[0], hi[1], hi[2], hi[3]);
                    st_shared_v4(b_lo(ks) + off, lo[0], lo[1], lo[2], lo[3]);
                }
            }
            fence_proxy_async_smem();
            __syncwarp();
            if (lane == 0) mbar_arrive(bres_bar);
        }
        if constexpr (NGRP == 1) {
            float va0[kChunks][4], vb0[kBIter][4], va1[kChunks][4], vb1[kBIter][4];
            if (nf > 0) load(va0, vb0);
            for (int f = 0; f < nf && ok; f += 2) {
                if (f + 1 < nf) load(va1, vb1);
                if (!store(f, va0, vb0)) { ok = false; break; }
                if (f + 1 < nf) {
                    if (f + 2 < nf) load(va0, vb0);
                    if (!store(f + 1, va1, vb1)) { ok = false; break; }
                }
            }
        } else {
            float va[kChunks][4], vb[kBIter][4];
            for (int f = grp; f < nf; f += NGRP) {
                load(va, vb);
                if (!store(f, va, vb)) break;
            }
        }
    } else if (warp == kMmaWarp && lane == 0) {
        // ---------------------------------------------------------- MMA issuer
        int stage = 0, slot = 0, acc = 0;
        uint32_t phase = 0, slot_phase = 0, acc_phase = 0;
        bool ok = true, any = false;
        if (RESB && (int)blockIdx.x < p.total_tiles)
            ok = mbar_wait(bres_bar, 0, abort_flag, p.status);   // the resident weights are split
        for (int tile = blockIdx.x; tile < p.total_tiles && ok; tile += gridDim.x) {
            if (!mbar_wait(corre_bar(acc), acc_phase ^ 1u, abort_flag, p.status)) { ok = false; break; }
            tc_fence_after();
            const uint32_t d_corr = tmem_base + (uint32_t)(acc * BN);
            for (int ks = 0; ks < p.KT; ++ks) {
                if (!mbar_wait(full_bar(stage), phase, abort_flag, p.status)) { ok = false; break; }
                TF_TRACE(1, 9);
                if (!mbar_wait(slote_bar(slot), slot_phase ^ 1u, abort_flag, p.status)) { ok = false; break; }
                TF_TRACE(1, 4);
                tc_fence_after();
                const uint32_t d_main = tmem_base + (uint32_t)(2 * BN + slot * BN);
                const uint64_t bh = smem_desc_sw128(b_hi(RESB ? ks : stage));
                const uint64_t bl = smem_desc_sw128(b_lo(RESB ? ks : stage));
                if constexpr (AT) {
                    // A in tensor memory: 8 columns per K step
                    const uint32_t ah = tmem_base + (uint32_t)(TM::kACol0 + stage * 64), al = ah + 32u;
#pragma unroll
                    for (int kk = 0; kk < kTfBK / 8; ++kk)
                        mma_tf32_ts(d_main, ah + (uint32_t)(kk * 8), bh + (uint64_t)(kk * 2), kIdesc,
                                    kk != 0 ? 1u : 0u);
#pragma unroll
                    for (int kk = 0; kk < kTfBK / 8; ++kk) {
                        const uint64_t o = (uint64_t)(kk * 2);
                        mma_tf32_ts(d_corr, ah + (uint32_t)(kk * 8), bl + o, kIdesc, (ks | kk) != 0 ? 1u : 0u);
                        mma_tf32_ts(d_corr, al + (uint32_t)(kk * 8), bh + o, kIdesc, 1u);
                    }
                } else {
                    const uint64_t ah = smem_desc_sw128(a_hi(stage)), al = smem_desc_sw128(a_lo(stage));
                    // advance 8 elements (32 bytes) along K inside the swizzled rows
#pragma unroll
                    for (int kk = 0; kk < kTfBK / 8; ++kk)
                        mma_tf32(d_main, ah + (uint64_t)(kk * 2), bh + (uint64_t)(kk * 2), kIdesc,
                                 kk != 0 ? 1u : 0u);
#pragma unroll
                    for (int kk = 0; kk < kTfBK / 8; ++kk) {
                        const uint64_t o = (uint64_t)(kk * 2);
                        mma_tf32(d_corr, ah + o, bl + o, kIdesc, (ks | kk) != 0 ? 1u : 0u);
                        mma_tf32(d_corr, al + o, bh + o, kIdesc, 1u);
                    }
                }
                any = true;
                TF_TRACE(1, 12);
                mma_commit(empty_bar(stage));
                mma_commit(slotf_bar(slot));
                if (++stage == STAGES) { stage = 0; phase ^= 1u; }
                if (++slot == kSlots) { slot = 0; slot_phase ^= 1u; }
            }
            if (!ok) break;
            mma_commit(corrf_bar(acc));
            if (++acc == 2) { acc = 0; acc_phase ^= 1u; }
        }
        if (any) {
            // every MMA must retire before tensor memory is released
            mma_commit(drain_bar);
            const long long t0 = clock64();
            while (!mbar_try_wait(drain_bar, 0) && cycles_left(t0)) {
            }
        }
    } else if (warp < kEpiWarps) {
        // ---------------------------------------------------------- epilogue
        // Thread = one output pixel (accumulator lane) x kCpt channels.  Per
        // stage: tcgen05.ld of the stage's x_hi*w_hi slot, fp32 adds into
        // registers; per tile: + the correction accumulator, + bias, store.
        // NCHW: a warp's 32 pixels are consecutive in y for each channel, so
        // every store instruction writes whole lines.
        const int quarter = warp & 3;
        const int col0 = (warp >> 2) * kCpt;
        const int row = quarter * 32 + lane;
        const uint32_t t_lane = tmem_base + ((uint32_t)(quarter * 32) << 16);
        int slot = 0, acc = 0;
        uint32_t slot_phase = 0, acc_phase = 0;
        bool ok = true;
        for (int tile = blockIdx.x; tile < p.total_tiles && ok; tile += gridDim.x) {
            // The sums start from the bias: its loads are issued together
            // here, while the tile's first stage is still being filled, and
            // none of them follows a store of this tile.  (The tile's
            // coordinates are computed again after the main loop, so that
            // only the sums stay live across it.)
            // column pairs (2i, 2i + 1), added as add.rn.f32x2 (two fp32 adds,
            // each rounded as a scalar add, per instruction)
            uint64_t a2[kCpt / 2];
            const int kb0 = (tile % p.n_tiles_n) * BN + col0;
#pragma unroll
            for (int j = 0; j < kCpt; j += 2) {
                float bv[2];
#pragma unroll
                for (int e = 0; e < 2; ++e) {
                    const int k = kb0 + j + e;
                    const int bk = LSTM ? (k & 3) * p.lstm_ch + (k >> 2) : k;
                    const bool bin = p.bias != nullptr && k < p.K;
                    bv[e] = ldg_or_zero(bin ? p.bias + bk : p.x, bin);
                }
                a2[j / 2] = pack_f32x2(bv[0], bv[1]);
            }
            for (int ks = 0; ks < p.KT; ++ks) {
                int okw = 1;
                if (lane == 0) okw = mbar_wait(slotf_bar(slot), slot_phase, abort_flag, p.status) ? 1 : 0;
                okw = __shfl_sync(0xffffffffu, okw, 0);
                if (!okw) { ok = false; break; }
                if (threadIdx.x == 0) TF_TRACE(2, 7);
                tc_fence_after();
#pragma unroll
                for (int c = 0; c < kCpt; c += 16) {
                    uint32_t v[16];
                    tmem_ld_16cols(t_lane + (uint32_t)(2 * BN + slot * BN + col0 + c), v);
#pragma unroll
                    for (int j = 0; j < 16; j += 2)
                        a2[(c + j) / 2] = fadd2(a2[(c + j) / 2], ((uint64_t)v[j + 1] << 32) | v[j]);
                }
                tc_fence_before();
                __syncwarp();
                if (lane == 0) mbar_arrive(slote_bar(slot));
                if (threadIdx.x == 0) TF_TRACE(2, 8);
                if (++slot == kSlots) { slot = 0; slot_phase ^= 1u; }
            }
            if (!ok) break;
            int okw = 1;
            if (lane == 0) okw = mbar_wait(corrf_bar(acc), acc_phase, abort_flag, p.status) ? 1 : 0;
            okw = __shfl_sync(0xffffffffu, okw, 0);
            if (!okw) break;
            if (threadIdx.x == 0) TF_TRACE(2, 10);
            tc_fence_after();
#pragma unroll
            for (int c = 0; c < kCpt; c += 16) {
                uint32_t v[16];
                tmem_ld_16cols(t_lane + (uint32_t)(acc * BN + col0 + c), v);
#pragma unroll
                for (int j = 0; j < 16; j += 2)
                    a2[(c + j) / 2] = fadd2(a2[(c + j) / 2], ((uint64_t)v[j + 1] << 32) | v[j]);
            }
            float a[kCpt];
#pragma unroll
            for (int j = 0; j < kCpt; j += 2) unpack_f32x2(a2[j / 2], a[j], a[j + 1]);
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(corre_bar(acc));
            if (++acc == 2) { acc = 0; acc_phase ^= 1u; }

            const int tm = tile / p.n_tiles_n;
            const int tn = tile - tm * p.n_tiles_n;
            const int64_t m = (int64_t)tm * kTfBM + row;
            const int kb = tn * BN + col0;
            if (m >= p.M) continue;
            if (LSTM) {
                // gates -> state update: c = f*c_prev + i*g, h = o*tanh(c)
                const int64_t n = m / p.PQ;
                const int64_t pq = m - n * p.PQ;
                const int Ch = p.lstm_ch;
                // the previous cell state of this pixel's hidden units, all
                // loaded before the first store
                float cp[kCpt / 4];
#pragma unroll
                for (int j = 0; j < kCpt; j += 4) {
                    const int u = (kb + j) >> 2;
                    cp[j / 4] = ldg_or_zero(p.c_prev + (u < Ch ? (n * Ch + u) * p.PQ + pq : 0), u < Ch);
                }
#pragma unroll
                for (int j = 0; j < kCpt; j += 4) {
                    const int u = (kb + j) >> 2;
                    if (u >= Ch) break;
                    const float ig = sigmoidf_(a[j]), fg = sigmoidf_(a[j + 1]), og = sigmoidf_(a[j + 2]);
                    const float gg = tanhf(a[j + 3]);
                    const int64_t ci = (n * Ch + u) * p.PQ + pq;
                    const float c = fg * cp[j / 4] + ig * gg;
                    p.c_next[ci] = c;
                    p.h_next[n * p.h_img + (int64_t)u * p.PQ + pq] = og * tanhf(c);
                }
            } else if (p.nhwc) {
                float *yr = p.y + m * p.K;
                if (p.y_vec) {
#pragma unroll
                    for (int j = 0; j < kCpt; j += 4) {
                        const int k = kb + j;
                        if (k < p.K) {
                            float4 o;
                            o.x = a[j];
                            o.y = a[j + 1];
                            o.z = a[j + 2];
                            o.w = a[j + 3];
                            *reinterpret_cast<float4 *>(yr + k) = o;
                        }
                    }
                } else {
#pragma unroll
                    for (int j = 0; j < kCpt; ++j) {
                        const int k = kb + j;
                        if (k < p.K) yr[k] = a[j];
                    }
                }
            } else {
                const int64_t n = m / p.PQ;
                float *yr;
                int64_t kst;
                if (p.dv) {
                    // output (a + st*i, b + st*j) of the residue class
                    const int rem = (int)(m - n * p.PQ);
                    const int i = rem / p.Q, jj = rem - i * p.Q;
                    kst = (int64_t)p.dv_H * p.dv_W;
                    yr = p.y + n * p.K * kst + (int64_t)(p.dv_a + p.dv_st * i) * p.dv_W + p.dv_b + p.dv_st * jj;
                } else {
                    kst = p.PQ;
                    yr = p.y + n * p.K * p.PQ + (m - n * p.PQ);
                }
#pragma unroll
                for (int j = 0; j < kCpt; ++j) {
                    const int k = kb + j;
                    if (k < p.K) yr[(int64_t)k * kst] = a[j];
                }
            }
            if (threadIdx.x == 0) TF_TRACE(2, 11);
        }
    }

    tc_fence_before();
    __syncthreads();
    if (warp == kMmaWarp) {
        __syncwarp();
        tc_fence_after();
        tmem_dealloc(tmem_base, TM::kCols);
    }
}

bool ensure_attr(const void *kern, size_t bytes, std::atomic<uint64_t> &done_mask) {
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

template <int BN, int STAGES, int NPROD, bool LSTM, bool RESB, int NGRP, bool AT>
conv2d_status_t launch_tf(const Shape &s, const Plan &pl, const Tensors &t, const TfLstm *lstm,
                          cudaStream_t st, const TfDeconv *dv = nullptr) {
    using L = TfSmem<BN, STAGES, RESB, AT>;
    TfParams p;
    p.x = static_cast<const float *>(t.x);
    p.w = static_cast<const float *>(t.w);
    p.bias = static_cast<const float *>(t.bias);
    p.y = static_cast<float *>(t.y);
    p.status = status_word_ptr();
    p.M = s.M;
    p.img = (int64_t)s.C * s.H * s.W;
    p.K = s.K;
    p.Kg = (int)s.Kg;
    p.KT = (int)((s.Kg + kTfBK - 1) / kTfBK);
    p.C = s.C;
    p.H = s.H;
    p.W = s.W;
    p.S = s.S;
    p.RS = s.R * s.S;
    p.Q = s.Q;
    p.PQ = s.P * s.Q;
    p.stride = s.stride;
    p.pad = s.pad;
    p.dil = s.dil;
    p.n_tiles_n = (s.K + BN - 1) / BN;
    const int64_t tiles = ((s.M + kTfBM - 1) / kTfBM) * (int64_t)p.n_tiles_n;
    if (tiles > INT32_MAX) return CONV2D_ERR_UNSUPPORTED;
    p.total_tiles = (int)tiles;
    p.nhwc = s.layout == CONV2D_NHWC ? 1 : 0;
    p.R = s.R;
    p.rs_mask = s.R * s.S <= 63 ? 1 : 0;
    p.tap4 = (s.layout == CONV2D_NCHW && s.R == 2 && s.S == 2) ? 1 : 0;
    p.HW = s.H * s.W;   // C*H*W < 2^31 (tf_shape_ok)
    p.dilW = s.dil * s.W;
    p.dv = 0;
    if (dv) {
        p.dv = 1;
        p.dv_H = dv->H; p.dv_W = dv->W; p.dv_a = dv->a; p.dv_b = dv->b; p.dv_st = dv->st;
        p.dv_J = dv->J; p.dv_L = dv->L; p.dv_R = dv->R; p.dv_S = dv->S;
        for (int i = 0; i < 8; ++i) {
            p.dv_e[i] = dv->e[i]; p.dv_f[i] = dv->f[i]; p.dv_r[i] = dv->r[i]; p.dv_s[i] = dv->s[i];
        }
        p.rs_mask = 0;
        p.tap4 = 0;
    }
    p.lstm_ch = 0;
    p.c_prev = nullptr;
    p.c_next = nullptr;
    p.h_next = nullptr;
    p.h_img = 0;
    if (LSTM) {
        if (!lstm || s.layout != CONV2D_NCHW || s.K % 4) return CONV2D_ERR_INTERNAL;
        p.lstm_ch = s.K / 4;
        p.c_prev = lstm->c_prev;
        p.c_next = lstm->c_next;
        p.h_next = lstm->h_next;
        p.h_img = lstm->h_img;
    }
    // float4 weight loads need contiguous weight rows: not the transposed
    // convolution's [K_in][K][R][S] layout
    p.w_vec = (!dv && s.Kg % 4 == 0 && ((uintptr_t)t.w & 15) == 0) ? 1 : 0;
    p.y_vec = (p.nhwc && s.K % 4 == 0 && ((uintptr_t)t.y & 15) == 0) ? 1 : 0;
    const size_t bytes = L::bytes(p.KT);
    auto kern = tf32x3_conv_kernel<BN, STAGES, NPROD, LSTM, RESB, NGRP, AT>;
    static std::atomic<uint64_t> attr_done{0};   // this instantiation's per-device flags
    // the attribute is set for the largest table this variant accepts
    if (!ensure_attr(reinterpret_cast<const void *>(kern), 227 * 1024, attr_done)) return CONV2D_ERR_CUDA;
    if (bytes > 227 * 1024) return CONV2D_ERR_UNSUPPORTED;
    int grid = pl.grid > 0 ? pl.grid : 1;
    if (RESB) {
        // every CTA must keep one output-channel tile: gridDim % n_tiles_n == 0
        grid = std::max(p.n_tiles_n, grid / p.n_tiles_n * p.n_tiles_n);
    }
    if (launch_pdl(kern, dim3(grid), dim3(tf_threads<BN, NPROD>()), bytes, st, p) != cudaSuccess) {
        cudaGetLastError();
        return CONV2D_ERR_CUDA;
    }
    return CONV2D_OK;
}

// Only variants with 8 or more producer warps carry the ConvLSTM epilogue.
template <int BN, int STAGES, int NPROD, bool RESB, int NGRP, bool AT>
conv2d_status_t launch_tf_lstm(const Shape &s, const Plan &pl, const Tensors &t, const TfLstm *lstm,
                               cudaStream_t st) {
    if constexpr (NPROD >= 8)
        return launch_tf<BN, STAGES, NPROD, true, RESB, NGRP, AT>(s, pl, t, lstm, st, nullptr);
    return CONV2D_ERR_UNSUPPORTED;
}

// (BN, STAGES, producer warps, measured ns per stage of one tile, resident
// weights, producer groups, A in tensor memory) of every compiled variant.  The stage times were measured on GB300 on the MSCRED
// encoder layers (fp32 NCHW, 3x3 / 2x2 filters); the producers' gather is
// latency-bound, so more producer warps per SM run a stage faster.  The
// 3-stage variant leaves shared memory for the tap tables of long
// reductions (C*R*S up to about 9,000).  The last three keep the split input
// in tensor memory (AT): correct, and measured within a few percent of their
// shared-memory siblings on the MSCRED encoder layers, so their costs are set
// just above those.  The resident-weight variants split
// the weights once per CTA (C*R*S up to about 350 at BN = 64).  Two producer
// groups (last four rows) took the encoder layers 5-10 % and the decoder's
// 32-channel-wide residue classes 7-14 % below the best one-group variant.
#define CONV2D_TF_VARIANTS(X)               \
    X(32, 5, 4, 1240, false, 1, false)      \
    X(64, 4, 4, 3850, false, 1, false)      \
    X(128, 3, 4, 5000, false, 1, false)     \
    X(32, 5, 8, 920, false, 1, false)       \
    X(64, 4, 8, 1370, false, 1, false)      \
    X(128, 3, 8, 3100, false, 1, false)     \
    X(64, 4, 16, 1100, false, 1, false)     \
    X(64, 3, 16, 1060, false, 1, false)     \
    X(64, 2, 16, 1060, true, 1, false)      \
    X(64, 3, 16, 1060, true, 1, false)      \
    X(64, 4, 16, 990, false, 2, false)      \
    X(64, 2, 16, 940, true, 2, false)       \
    X(128, 2, 16, 2400, false, 2, false)    \
    X(32, 5, 16, 820, false, 2, false)      \
    X(64, 4, 16, 1000, true, 2, true)       \
    X(64, 4, 16, 1000, false, 2, true)      \
    X(32, 4, 16, 830, false, 2, true)

}  // namespace

// Variants compiled with the ConvLSTM-cell epilogue: 8 and 16 producer warps.
bool tf_lstm_variant(int id) { return tf_variant(id).nprod >= 8; }

int tf_num_variants() {
    int n = 0;
#define X(vbn, vst, vnp, vns, vrb, vng, vat) ++n;
    CONV2D_TF_VARIANTS(X)
#undef X
    return n;
}

TfTile tf_variant(int id) {
    int i = 0;
    TfTile t{0, 0, 0, -1, 0, false, 1, false};
#define X(vbn, vst, vnp, vns, vrb, vng, vat)                        \
    if (i == id) t = TfTile{vbn, vst, vnp, id, vns, vrb, vng, vat}; \
    ++i;
    CONV2D_TF_VARIANTS(X)
#undef X
    return t;
}

size_t tf_smem_bytes(const Shape &s, const TfTile &t) {
    const size_t kt = (size_t)((s.Kg + kTfBK - 1) / kTfBK);
    const size_t btile = (size_t)t.BN * kTfBK * 4;
    const size_t stage = (t.at ? 0 : 2 * (size_t)kTfATile) + (t.resb ? 0 : 2 * btile);
    size_t slots = t.BN >= 128 ? 2 : 6;
    if (t.at) {
        const size_t fr = (512 - 2 * (size_t)t.BN - 64 * (size_t)t.stages) / t.BN;
        slots = fr > 6 ? 6 : fr;
    }
    const size_t bars = (2 * (size_t)t.stages + 2 * slots + 6) * 8;
    const size_t end = (size_t)t.stages * stage + bars + 16;
    const size_t taps = t.resb ? (end + 1023) / 1024 * 1024 + kt * 2 * btile : (end + 15) / 16 * 16;
    return taps + kt * kTfBK * 12 + 1024;
}

bool tf_shape_ok(const Shape &s) {
    if (s.dtype != CONV2D_F32) return false;
    if (s.H > 32767 || s.W > 32767) return false;
    if ((int64_t)s.dil * (s.R - 1) > 32767 || (int64_t)s.dil * (s.S - 1) > 32767) return false;
    if (s.Kg > ((int64_t)1 << 20)) return false;
    // 32-bit tap offsets within one image
    const int64_t span_h = (int64_t)s.dil * (s.R - 1) + 1, span_w = (int64_t)s.dil * (s.S - 1) + 1;
    const int64_t lim = (int64_t)1 << 31;
    if ((int64_t)s.C * s.H * s.W >= lim) return false;
    if ((span_h * s.W + span_w) * s.C >= lim) return false;
    if ((int64_t)s.C * s.H * s.W + span_h * s.W + span_w >= lim) return false;
    if ((int64_t)s.P * s.Q >= lim) return false;
    return true;
}

#ifdef CONV2D_TC_TRACE
extern "C" int conv2d_tf_trace_dump(unsigned long long *out, unsigned int *counts) {
    if (cudaDeviceSynchronize() != cudaSuccess) return -1;
    if (cudaMemcpyFromSymbol(counts, g_tf_trace_n, sizeof(unsigned int) * 4) != cudaSuccess) return -1;
    if (cudaMemcpyFromSymbol(out, g_tf_trace, sizeof(unsigned long long) * 4 * 8192) != cudaSuccess) return -1;
    const unsigned int zero[4] = {0, 0, 0, 0};
    return cudaMemcpyToSymbol(g_tf_trace_n, zero, sizeof(zero)) == cudaSuccess ? 0 : -1;
}
#endif

conv2d_status_t tf_launch(const Shape &s, const Plan &pl, const Tensors &t, cudaStream_t st,
                          const TfLstm *lstm, const TfDeconv *dv) {
    int i = 0;
#define X(vbn, vst, vnp, vns, vrb, vng, vat)                                                    \
    if (pl.tf.id == i) {                                                                        \
        if (dv) return launch_tf<vbn, vst, vnp, false, vrb, vng, vat>(s, pl, t, nullptr, st, dv); \
        if (lstm) return launch_tf_lstm<vbn, vst, vnp, vrb, vng, vat>(s, pl, t, lstm, st);      \
        return launch_tf<vbn, vst, vnp, false, vrb, vng, vat>(s, pl, t, nullptr, st);            \
    }                                                                                           \
    ++i;
    CONV2D_TF_VARIANTS(X)
#undef X
    return CONV2D_ERR_INTERNAL;
}

}  // namespace conv2d
