// Device status word: kernels that give up on a bounded barrier wait record
// the failure here instead of trapping, so the CUDA context stays usable and
// the host can read the reason with conv2d_get_device_status().

#include <mutex>

#include "internal.h"

namespace conv2d {

__device__ unsigned int g_status_word = 0;

namespace {
constexpr int kMaxDevices = 64;
std::mutex g_mu;
unsigned int *g_ptr[kMaxDevices] = {};
}  // namespace

unsigned int *status_word_ptr() {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return nullptr;
    std::lock_guard<std::mutex> lk(g_mu);
    if (!g_ptr[dev]) {
        void *p = nullptr;
        if (cudaGetSymbolAddress(&p, g_status_word) != cudaSuccess) return nullptr;
        g_ptr[dev] = static_cast<unsigned int *>(p);
    }
    return g_ptr[dev];
}

conv2d_status_t status_read_and_clear() {
    if (cudaDeviceSynchronize() != cudaSuccess) return CONV2D_ERR_CUDA;
    unsigned int v = 0, zero = 0;
    if (cudaMemcpyFromSymbol(&v, g_status_word, sizeof(v)) != cudaSuccess) return CONV2D_ERR_CUDA;
    if (v != 0 && cudaMemcpyToSymbol(g_status_word, &zero, sizeof(zero)) != cudaSuccess)
        return CONV2D_ERR_CUDA;
    return v == 0 ? CONV2D_OK : CONV2D_ERR_TIMEOUT;
}

}  // namespace conv2d
