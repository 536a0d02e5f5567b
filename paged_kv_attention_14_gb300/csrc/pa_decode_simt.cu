// pa_decode_simt.cu -- instantiations of the CUDA-core decode kernel
// (group sizes 1, 2 and 4; head_dim 64 and 128; bf16, fp16, E4M3 and E5M2
// caches).
#include "pa_decode_kernels.cuh"

namespace pa {
namespace dec {

template <int D, int KVT>
static KernelInfo simt_for(int g) {
  if (g <= 1) return simt_info<D, KVT, 1>();
  if (g <= 2) return simt_info<D, KVT, 2>();
  return simt_info<D, KVT, 4>();
}

template <int D>
static KernelInfo simt_for_dtype(int kv_dtype, int g) {
  if (kv_dtype == PA_KV_BF16) return simt_for<D, kKvBf16>(g);
  if (kv_dtype == PA_KV_F16) return simt_for<D, kKvF16>(g);
  if (kv_dtype == PA_KV_FP8_E5M2) return simt_for<D, kKvE5M2>(g);
  return simt_for<D, kKvFp8>(g);
}

KernelInfo pick_simt(int head_dim, int kv_dtype, int g) {
  return head_dim == 128 ? simt_for_dtype<128>(kv_dtype, g) : simt_for_dtype<64>(kv_dtype, g);
}

}  // namespace dec
}  // namespace pa
