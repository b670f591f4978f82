// Throughput probes: kernels that do nothing but FFMAs or tensor-core MMAs on
// on-chip operands, so that a caller timing one launch with CUDA events gets
// the GPU's attainable fp32 FFMA, TF32 and BF16 MMA rates.  They give the
// roofline denominators of the fp32 kernels (FFMA for the direct / implicit
// GEMM kernels, TF32 for the 3xTF32 kernel) a measured value beside the
// separately measured HBM copy bandwidth and cuBLAS BF16 throughput.

#include <cuda.h>

#include <atomic>

#include "internal.h"
#include "ptx_sm103a.cuh"

namespace conv2d {
namespace {

using namespace sm103a;

// Sink for the FFMA results: written only if a sum equals a value no chain
// reaches, so the chains cannot be removed as dead code.
__device__ float g_probe_sink;

constexpr int kFfmaChains = 16;
constexpr int kFfmaThreads = 256;

__global__ void __launch_bounds__(kFfmaThreads) ffma_probe_kernel(int iters, float seed) {
    float a[kFfmaChains];
#pragma unroll
    for (int i = 0; i < kFfmaChains; ++i) a[i] = seed + (float)(threadIdx.x + i);
    const float m = 0.999999f, c = 1e-7f;
    for (int it = 0; it < iters; ++it) {
#pragma unroll
        for (int u = 0; u < 8; ++u) {
#pragma unroll
            for (int i = 0; i < kFfmaChains; ++i) a[i] = fmaf(a[i], m, c);
        }
    }
    float s = 0.f;
#pragma unroll
    for (int i = 0; i < kFfmaChains; ++i) s += a[i];
    if (s == -1.2345f) g_probe_sink = s;
}

// One CTA per SM; one thread issues `iters` x 4 MMAs (M=128, N=256) on
// zero-filled operands in shared memory into one tensor-memory accumulator,
// then waits for them to retire.  kind::tf32 takes K=8 per MMA, kind::f16
// (bf16 operands) K=16; both read 128-byte K-major swizzled rows.
constexpr int kMmaN = 256;
constexpr int kMmaThreads = 128;
constexpr int kATile = 128 * 128;     // 128 rows x 128 bytes
constexpr int kBTile = kMmaN * 128;   // 256 rows x 128 bytes
// More than half of an SM's shared memory, so that no two probe CTAs share an SM.
constexpr int kMmaSmem = 120 * 1024;
static_assert(kATile + kBTile + 1024 + 64 <= kMmaSmem, "probe shared memory");

__device__ __forceinline__ void probe_mma(bool tf32, uint32_t d, uint64_t a, uint64_t b, uint32_t idesc,
                                          uint32_t acc) {
    if (tf32)
        asm volatile(
            "{\n\t.reg .pred p;\n\tsetp.ne.b32 p, %4, 0;\n\t"
            "tcgen05.mma.cta_group::1.kind::tf32 [%0], %1, %2, %3, p;\n\t}" ::"r"(d),
            "l"(a), "l"(b), "r"(idesc), "r"(acc)
            : "memory");
    else
        asm volatile(
            "{\n\t.reg .pred p;\n\tsetp.ne.b32 p, %4, 0;\n\t"
            "tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n\t}" ::"r"(d),
            "l"(a), "l"(b), "r"(idesc), "r"(acc)
            : "memory");
}

__global__ void __launch_bounds__(kMmaThreads, 1) mma_probe_kernel(int iters, int tf32, unsigned int *status) {
    extern __shared__ uint8_t smem_raw[];
    uint8_t *smem = smem_raw + ((1024u - (smem_u32(smem_raw) & 1023u)) & 1023u);
    const uint32_t base = smem_u32(smem);
    const uint32_t a_s = base, b_s = base + kATile;
    const uint32_t bar = base + kATile + kBTile;
    uint32_t *tmem_holder = reinterpret_cast<uint32_t *>(smem + kATile + kBTile + 8);
    volatile int *abort_flag = reinterpret_cast<volatile int *>(smem + kATile + kBTile + 12);
    const int warp = threadIdx.x / 32;
    for (int i = threadIdx.x; i < (kATile + kBTile) / 16; i += blockDim.x)
        st_shared_v4(base + 16u * i, 0u, 0u, 0u, 0u);
    if (threadIdx.x == 0) {
        mbar_init(bar, 1);
        *abort_flag = 0;
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    }
    fence_proxy_async_smem();
    if (warp == 0) {
        tmem_alloc(smem_u32(tmem_holder), kMmaN);
        tmem_relinquish();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *tmem_holder;
    if (threadIdx.x == 0) {
        // kind::tf32: A/B format 2; kind::f16 with bf16 operands: format 1
        const uint32_t fmt = tf32 ? 2u : 1u;
        const uint32_t idesc = (1u << 4) | (fmt << 7) | (fmt << 10) | ((uint32_t)(kMmaN >> 3) << 17) |
                               ((uint32_t)(128 >> 4) << 24);
        const uint64_t ad = smem_desc_sw128(a_s), bd = smem_desc_sw128(b_s);
        for (int it = 0; it < iters; ++it) {
#pragma unroll
            for (int k = 0; k < 4; ++k)   // four K steps span one 128-byte row
                probe_mma(tf32 != 0, tmem, ad + (uint64_t)(k * 2), bd + (uint64_t)(k * 2), idesc,
                          (it | k) != 0 ? 1u : 0u);
        }
        mma_commit(bar);
        mbar_wait(bar, 0, abort_flag, status);
    }
    tc_fence_before();
    __syncthreads();
    if (warp == 0) {
        tc_fence_after();
        tmem_dealloc(tmem, kMmaN);
    }
}

}  // namespace
}  // namespace conv2d

using namespace conv2d;

extern "C" conv2d_status_t conv2d_peak_probe(conv2d_peak_kind_t kind, int iters, cudaStream_t stream,
                                             double *flops) {
    if (!flops || iters < 1 || iters > (1 << 24)) return CONV2D_ERR_INVALID_ARG;
    int dev = 0, sms = 0, major = 0, minor = 0;
    if (cudaGetDevice(&dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, dev) != cudaSuccess)
        return CONV2D_ERR_CUDA;
    if (kind == CONV2D_PEAK_FFMA) {
        const int blocks = sms * 8;   // 2048 threads per SM
        ffma_probe_kernel<<<blocks, kFfmaThreads, 0, stream>>>(iters, 1.0f);
        if (cudaGetLastError() != cudaSuccess) return CONV2D_ERR_CUDA;
        *flops = 2.0 * kFfmaChains * 8.0 * iters * (double)blocks * kFfmaThreads;
        return CONV2D_OK;
    }
    if (kind != CONV2D_PEAK_TF32_MMA && kind != CONV2D_PEAK_BF16_MMA) return CONV2D_ERR_INVALID_ARG;
    if (!(major == 10 && minor == 3)) return CONV2D_ERR_UNSUPPORTED;
    // the attribute once per device: setting it on every call stalls the host
    // between the caller's timing events
    static std::atomic<uint64_t> attr_done{0};
    const uint64_t bit = (uint64_t)1 << (dev & 63);
    if (!(attr_done.load(std::memory_order_acquire) & bit)) {
        if (cudaFuncSetAttribute(mma_probe_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, kMmaSmem) !=
            cudaSuccess)
            return CONV2D_ERR_CUDA;
        attr_done.fetch_or(bit, std::memory_order_release);
    }
    const int tf32 = kind == CONV2D_PEAK_TF32_MMA ? 1 : 0;
    mma_probe_kernel<<<sms, kMmaThreads, kMmaSmem, stream>>>(iters, tf32, status_word_ptr());
    if (cudaGetLastError() != cudaSuccess) return CONV2D_ERR_CUDA;
    const double k = tf32 ? 8.0 : 16.0;
    *flops = 2.0 * 128.0 * kMmaN * k * 4.0 * iters * (double)sms;
    return CONV2D_OK;
}
