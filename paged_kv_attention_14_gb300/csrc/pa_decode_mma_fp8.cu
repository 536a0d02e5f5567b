// pa_decode_mma_fp8.cu -- instantiations of the tensor-core decode kernel
// for E4M3 caches: head_dim 64 and 128, groups of up to 4, 8 or 16 query
// heads per kv head, 1 or 2 kv heads per stage.
#include "pa_decode_kernels.cuh"

namespace pa {
namespace dec {

KernelInfo pick_mma_fp8(int head_dim, int gq, int hg) {
  return head_dim == 128 ? fp8_mma_for<kKvFp8, 128>(gq, hg) : fp8_mma_for<kKvFp8, 64>(gq, hg);
}

}  // namespace dec
}  // namespace pa
