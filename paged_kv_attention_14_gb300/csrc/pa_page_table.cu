// pa_page_table.cu -- prefix-cache page bookkeeping on the device.
//
// A radix-tree prefix cache maps token prefixes to physical pages of the
// block-paged KV pool ("1. Technical Mechanics of the Radix Cache" of
// "Building and Deploying vllm.cpp ..."):
//  * a hit binds the new sequence's block table directly to the pages its
//    matched prefix already occupies ("Zero-Copy Cache Hits"), and every
//    bound page gains one owner;
//  * when a sequence finishes or the cache evicts an entry ("LRU Eviction")
//    each of its pages loses one owner, and a page left without owners goes
//    back to the global page pool.
// The tree, the LRU order and the choice of what to evict are host logic;
// the page-table writes and the owner counts live on the device next to
// the cache, so a step never waits for a host copy of them.
//
// One CTA per sequence; its threads walk the sequence's pages.  Owner
// counts change by atomics, so several sequences may bind or release the
// same page in one call.  Page ids, table rows and hit lengths are always
// range-checked (these kernels are latency-bound; the checks are free):
// an entry outside the pool or the table is skipped and reported.
#include "pa_device.cuh"
#include "pa_internal.h"

namespace pa {

namespace {

constexpr int kThreads = 128;

__global__ void __launch_bounds__(kThreads) bind_blocks_kernel(int32_t *__restrict__ block_tables,
                                                               int max_blocks_per_seq, int num_rows,
                                                               const int32_t *__restrict__ seq_rows,
                                                               const int32_t *__restrict__ hit_start,
                                                               const int32_t *__restrict__ hit_blocks,
                                                               int32_t *__restrict__ refcounts, int num_blocks,
                                                               int32_t *err) {
  const int i = blockIdx.x;
  const int row = __ldg(seq_rows + i);
  const int h0 = __ldg(hit_start + i);
  const int n = __ldg(hit_start + i + 1) - h0;
  if (row < 0 || row >= num_rows || n < 0 || n > max_blocks_per_seq) {
    if (threadIdx.x == 0) report_error(err, nullptr, kErrBadIndex);
    return;
  }
  int32_t *trow = block_tables + static_cast<int64_t>(row) * max_blocks_per_seq;
  for (int j = threadIdx.x; j < n; j += kThreads) {
    const int blk = __ldg(hit_blocks + h0 + j);
    if (blk < 0 || blk >= num_blocks) {
      report_error(err, nullptr, kErrBadIndex);
      continue;
    }
    trow[j] = blk;
    atomicAdd(refcounts + blk, 1);
  }
}

__global__ void __launch_bounds__(kThreads) release_blocks_kernel(int32_t *__restrict__ block_tables,
                                                                  int max_blocks_per_seq, int num_rows,
                                                                  const int32_t *__restrict__ seq_rows,
                                                                  const int32_t *__restrict__ block_counts,
                                                                  int32_t *__restrict__ refcounts, int num_blocks,
                                                                  int32_t *__restrict__ free_list,
                                                                  int32_t *__restrict__ free_count, int32_t *err) {
  const int i = blockIdx.x;
  const int row = __ldg(seq_rows + i);
  const int n = __ldg(block_counts + i);
  if (row < 0 || row >= num_rows || n < 0 || n > max_blocks_per_seq) {
    if (threadIdx.x == 0) report_error(err, nullptr, kErrBadIndex);
    return;
  }
  int32_t *trow = block_tables + static_cast<int64_t>(row) * max_blocks_per_seq;
  for (int j = threadIdx.x; j < n; j += kThreads) {
    const int blk = trow[j];
    if (blk < 0 || blk >= num_blocks) {
      report_error(err, nullptr, kErrBadIndex);
      continue;
    }
    const int before = atomicSub(refcounts + blk, 1);
    if (before <= 0) {
      // no owner left to release: undo, report, leave the entry
      atomicAdd(refcounts + blk, 1);
      report_error(err, nullptr, kErrRefcount);
      continue;
    }
    trow[j] = -1;
    if (before == 1) {
      // the last owner left: the page returns to the pool (each page at
      // most once per owner count reaching zero)
      const int slot = atomicAdd(free_count, 1);
      if (slot >= 0 && slot < num_blocks)
        free_list[slot] = blk;
      else
        report_error(err, nullptr, kErrBadIndex);
    }
  }
}

}  // namespace

cudaError_t launch_bind_blocks(const pa_kv_desc &d, int32_t *block_tables, int32_t max_blocks_per_seq,
                               int32_t num_rows, const int32_t *seq_rows, const int32_t *hit_start,
                               const int32_t *hit_blocks, int32_t num_seqs, int32_t *refcounts, cudaStream_t stream) {
  bind_blocks_kernel<<<num_seqs, kThreads, 0, stream>>>(block_tables, max_blocks_per_seq, num_rows, seq_rows, hit_start,
                                                        hit_blocks, refcounts, d.num_blocks, d.error_word);
  return cudaGetLastError();
}

cudaError_t launch_release_blocks(const pa_kv_desc &d, int32_t *block_tables, int32_t max_blocks_per_seq,
                                  int32_t num_rows, const int32_t *seq_rows, const int32_t *block_counts,
                                  int32_t num_seqs, int32_t *refcounts, int32_t *free_list, int32_t *free_count,
                                  cudaStream_t stream) {
  release_blocks_kernel<<<num_seqs, kThreads, 0, stream>>>(block_tables, max_blocks_per_seq, num_rows, seq_rows,
                                                           block_counts, refcounts, d.num_blocks, free_list,
                                                           free_count, d.error_word);
  return cudaGetLastError();
}

}  // namespace pa
