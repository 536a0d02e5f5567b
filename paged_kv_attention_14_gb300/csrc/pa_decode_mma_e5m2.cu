// pa_decode_mma_e5m2.cu -- instantiations of the tensor-core decode kernel
// for E5M2 caches (the E4M3 kernel with an exact E5M2 -> f16 conversion):
// head_dim 64 and 128, groups of up to 4, 8 or 16 query heads per kv head,
// 1 or 2 kv heads per stage.
#include "pa_decode_kernels.cuh"

namespace pa {
namespace dec {

KernelInfo pick_mma_e5m2(int head_dim, int gq, int hg) {
  return head_dim == 128 ? fp8_mma_for<kKvE5M2, 128>(gq, hg) : fp8_mma_for<kKvE5M2, 64>(gq, hg);
}

}  // namespace dec
}  // namespace pa
