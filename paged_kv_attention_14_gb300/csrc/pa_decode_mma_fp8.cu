// pa_decode_mma_fp8.cu -- instantiations of the tensor-core decode kernel
// for E4M3 caches: head_dim 64 and 128, groups of up to 4, 8 or 16 query
// heads per kv head, 1 or 2 kv heads per stage.
#include "pa_decode_kernels.cuh"

namespace pa {
namespace dec {

// 8 consumer warps (see mma_info) while their partial-state buffers leave
// room for enough stages (up to 8 query heads per kv head), else 4;
// kv-head groups of 2 or 1
template <int GQ>
constexpr int fp8_consumer_warps() {
  return GQ <= 8 ? 8 : 4;
}

template <int D, int GQ>
static KernelInfo mma_for_hg(int hg) {
  if (hg >= 2) return mma_info<D, kKvFp8, GQ, 2, fp8_consumer_warps<GQ>()>();
  return mma_info<D, kKvFp8, GQ, 1, fp8_consumer_warps<GQ>()>();
}

template <int D>
static KernelInfo mma_for(int gq, int hg) {
  if (gq <= 4) return mma_for_hg<D, 4>(hg);
  if (gq <= 8) return mma_for_hg<D, 8>(hg);
  return mma_for_hg<D, 16>(hg);
}

KernelInfo pick_mma_fp8(int head_dim, int gq, int hg) {
  return head_dim == 128 ? mma_for<128>(gq, hg) : mma_for<64>(gq, hg);
}

}  // namespace dec
}  // namespace pa
