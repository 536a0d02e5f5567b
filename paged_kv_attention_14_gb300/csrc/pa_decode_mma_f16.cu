// pa_decode_mma_f16.cu -- instantiations of the tensor-core decode kernel
// for fp16 caches: head_dim 64 and 128, groups of up to 4, 8 or 16 query
// heads per kv head, 1, 2 or 4 kv heads per stage.
#include "pa_decode_kernels.cuh"

namespace pa {
namespace dec {

template <int D, int GQ>
static KernelInfo mma_for_hg(int hg) {
  if (hg >= 4) return mma_info<D, kKvF16, GQ, 4>();
  if (hg >= 2) return mma_info<D, kKvF16, GQ, 2>();
  return mma_info<D, kKvF16, GQ, 1>();
}

template <int D>
static KernelInfo mma_for(int gq, int hg) {
  if (gq <= 4) return mma_for_hg<D, 4>(hg);
  if (gq <= 8) return mma_for_hg<D, 8>(hg);
  return mma_for_hg<D, 16>(hg);
}

KernelInfo pick_mma_f16(int head_dim, int gq, int hg) {
  return head_dim == 128 ? mma_for<128>(gq, hg) : mma_for<64>(gq, hg);
}

}  // namespace dec
}  // namespace pa
