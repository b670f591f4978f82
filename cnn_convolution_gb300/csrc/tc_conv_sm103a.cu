// Tensor-core path placeholder (replaced by the tcgen05 kernel).
#include "internal.h"
namespace conv2d {
bool tc_shape_ok(const Shape &, const Tensors *) { return false; }
size_t tc_smem_bytes(const TcTile &) { return 0; }
conv2d_status_t tc_launch(const Shape &, const Plan &, const Tensors &, cudaStream_t) {
    return CONV2D_ERR_UNSUPPORTED;
}
}  // namespace conv2d
