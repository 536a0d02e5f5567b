// pa_cache_write.cu -- slot-mapped write of new K/V rows into the paged cache.
//
// The engine writes each new token's K/V into the physical block slot that
// the scheduler assigned to it (an indexed scatter through a slot mapping:
// "Block-Paged KV Cache (FP8/FP16)" in the architecture figure of "Building
// and Deploying vllm.cpp ...", and the device-resident indexed gather/scatter
// of the vllm.cpp status notes).  FP8 pages hold one byte per element
// ("2. CLI Configuration Parameters", --kv-cache-dtype fp8).
//
// One thread moves one 16-byte vector of a cache row: 8 bf16 / fp16 values
// (16 source bytes), or 16 values of an 8-bit cache (32 source bytes
// quantised to 16 bytes).  Consecutive threads cover consecutive vectors of
// a (token, kv head) row, so loads and stores are 16-byte vectorised and
// coalesced.  Negative slots are skipped; with checked indices a slot past
// the pool is skipped and reported.
#include "pa_device.cuh"
#include "pa_internal.h"

namespace pa {

template <int KVT>
__global__ void __launch_bounds__(256) cache_write_kernel(
    const uint4 *__restrict__ k, const uint4 *__restrict__ v, uint8_t *__restrict__ k_cache,
    uint8_t *__restrict__ v_cache, const int64_t *__restrict__ slot_mapping, int64_t total_vecs,
    int vecs_per_row, int num_kv_heads, int block_size, float k_scale, float v_scale,
    const float *__restrict__ k_scales, const float *__restrict__ v_scales, int64_t num_slots, int checked,
    int32_t *err) {
  // a kernel launched after this one as a programmatic dependent (pa_decode,
  // pa_prefill_chunk) may start its launch now; it waits for this grid's
  // writes before reading anything
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
  const int64_t i = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x;
  if (i >= total_vecs) return;
  const int vec = static_cast<int>(i % vecs_per_row);
  const int64_t row = i / vecs_per_row;  // token * num_kv_heads + head
  const int64_t token = row / num_kv_heads;
  const int head = static_cast<int>(row % num_kv_heads);
  const int64_t slot = __ldg(slot_mapping + token);
  if (slot < 0) return;
  if (checked && slot >= num_slots) {
    if (vec == 0) report_error(err, nullptr, kErrBadIndex);
    return;
  }
  const int64_t blk = slot / block_size;
  const int64_t off = slot % block_size;
  // destination row (blk, head, off) of [num_blocks][num_kv_heads][block_size][D]
  const int64_t dst = ((blk * num_kv_heads + head) * block_size + off) * vecs_per_row + vec;
  if constexpr (kv16(KVT)) {
    reinterpret_cast<uint4 *>(k_cache)[dst] = __ldg(k + i);
    reinterpret_cast<uint4 *>(v_cache)[dst] = __ldg(v + i);
  } else {
    // 16 values per store (encode_fp8x16); per-kv-head scales where given
    const float ks = k_scales ? __ldg(k_scales + head) : k_scale;
    const float vs = v_scales ? __ldg(v_scales + head) : v_scale;
    reinterpret_cast<uint4 *>(k_cache)[dst] = encode_fp8x16<KVT>(__ldg(k + 2 * i), __ldg(k + 2 * i + 1), ks);
    reinterpret_cast<uint4 *>(v_cache)[dst] = encode_fp8x16<KVT>(__ldg(v + 2 * i), __ldg(v + 2 * i + 1), vs);
  }
}

cudaError_t launch_cache_write(const pa_kv_desc &d, const void *k, const void *v, void *k_cache,
                               void *v_cache, const int64_t *slot_mapping, int32_t num_tokens,
                               cudaStream_t stream) {
  const bool b16 = d.kv_dtype == PA_KV_BF16 || d.kv_dtype == PA_KV_F16;
  const int vecs_per_row = d.head_dim / (b16 ? 8 : 16);  // 16-byte cache vectors per row
  const int64_t total = static_cast<int64_t>(num_tokens) * d.num_kv_heads * vecs_per_row;
  const int threads = 256;
  const int64_t blocks = (total + threads - 1) / threads;
  const float ks = d.k_scale == 0.f ? 1.f : d.k_scale;
  const float vs = d.v_scale == 0.f ? 1.f : d.v_scale;
  const int64_t num_slots = static_cast<int64_t>(d.num_blocks) * d.block_size;
  auto kern = b16 ? &cache_write_kernel<kKvBf16>  // 16-bit: bit copies
              : d.kv_dtype == PA_KV_FP8_E5M2 ? &cache_write_kernel<kKvE5M2>
                                             : &cache_write_kernel<kKvFp8>;
  kern<<<static_cast<unsigned>(blocks), threads, 0, stream>>>(
      static_cast<const uint4 *>(k), static_cast<const uint4 *>(v), static_cast<uint8_t *>(k_cache),
      static_cast<uint8_t *>(v_cache), slot_mapping, total, vecs_per_row, d.num_kv_heads, d.block_size, ks, vs,
      d.k_scales, d.v_scales, num_slots, d.check_indices, d.error_word);
  return cudaGetLastError();
}

}  // namespace pa
