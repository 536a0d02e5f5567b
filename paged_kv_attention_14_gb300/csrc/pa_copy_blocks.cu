// pa_copy_blocks.cu -- copy-on-write of whole pages of the paged cache.
//
// A prefix-cache hit binds a new sequence's block table to pages that other
// sequences already use ("Zero-Copy Cache Hits" of "1. Technical Mechanics of
// the Radix Cache", Building and Deploying vllm.cpp).  Before a sequence
// writes into such a page (the partly filled last page of the shared
// prefix), the engine gives it a private copy: block dst_blocks[i] of both
// caches receives block src_blocks[i], every kv head and slot.
//
// One thread moves one 16-byte vector of K and one of V; consecutive threads
// cover consecutive bytes of a block, so both the reads and the writes are
// coalesced 16-byte accesses.  With checked indices a pair naming a block
// outside the cache is skipped and reported.
#include "pa_device.cuh"
#include "pa_internal.h"

namespace pa {

__global__ void __launch_bounds__(256) copy_blocks_kernel(uint4 *__restrict__ k_cache, uint4 *__restrict__ v_cache,
                                                          const int32_t *__restrict__ src_blocks,
                                                          const int32_t *__restrict__ dst_blocks,
                                                          int64_t vecs_per_block, int64_t total_vecs,
                                                          int num_blocks, int checked, int32_t *err) {
  // a programmatic dependent launched after this one waits for these writes
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
  for (int64_t i = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x; i < total_vecs;
       i += static_cast<int64_t>(gridDim.x) * blockDim.x) {
    const int64_t pair = i / vecs_per_block;
    const int64_t off = i - pair * vecs_per_block;
    const int sb = __ldg(src_blocks + pair), db = __ldg(dst_blocks + pair);
    if (checked && (sb < 0 || sb >= num_blocks || db < 0 || db >= num_blocks)) {
      // checked indices: a pair naming a block outside the cache is skipped
      if (off == 0) report_error(err, nullptr, kErrBadIndex);
      continue;
    }
    const int64_t src = static_cast<int64_t>(sb) * vecs_per_block + off;
    const int64_t dst = static_cast<int64_t>(db) * vecs_per_block + off;
    k_cache[dst] = k_cache[src];
    v_cache[dst] = v_cache[src];
  }
}

cudaError_t launch_copy_blocks(const pa_kv_desc &d, void *k_cache, void *v_cache, const int32_t *src_blocks,
                               const int32_t *dst_blocks, int32_t num_pairs, cudaStream_t stream) {
  const int esz = (d.kv_dtype == PA_KV_BF16 || d.kv_dtype == PA_KV_F16) ? 2 : 1;
  const int64_t block_bytes = static_cast<int64_t>(d.num_kv_heads) * d.block_size * d.head_dim * esz;
  const int64_t vecs = block_bytes / 16;
  const int64_t total = vecs * num_pairs;
  const int threads = 256;
  // at most a few waves of the SMs; the loop strides over the rest
  const int64_t want = (total + threads - 1) / threads;
  const int64_t cap = static_cast<int64_t>(device_sm_count()) * 8;
  const unsigned blocks = static_cast<unsigned>(want < cap ? want : cap);
  copy_blocks_kernel<<<blocks, threads, 0, stream>>>(static_cast<uint4 *>(k_cache), static_cast<uint4 *>(v_cache),
                                                     src_blocks, dst_blocks, vecs, total, d.num_blocks,
                                                     d.check_indices, d.error_word);
  return cudaGetLastError();
}

}  // namespace pa
