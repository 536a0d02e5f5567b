// pa_decode_simt.cu -- instantiations of the CUDA-core decode kernel
// (group sizes 1, 2 and 4; head_dim 64 and 128; bf16 and E4M3 caches).
#include "pa_decode_kernels.cuh"

namespace pa {
namespace dec {

template <int D, int KVT>
static KernelInfo simt_for(int g) {
  if (g <= 1) return simt_info<D, KVT, 1>();
  if (g <= 2) return simt_info<D, KVT, 2>();
  return simt_info<D, KVT, 4>();
}

KernelInfo pick_simt(int head_dim, int kv_dtype, int g) {
  if (head_dim == 128) return kv_dtype == PA_KV_BF16 ? simt_for<128, kKvBf16>(g) : simt_for<128, kKvFp8>(g);
  return kv_dtype == PA_KV_BF16 ? simt_for<64, kKvBf16>(g) : simt_for<64, kKvFp8>(g);
}

}  // namespace dec
}  // namespace pa
