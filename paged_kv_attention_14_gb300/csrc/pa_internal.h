// pa_internal.h -- launchers shared between the C-ABI layer and the kernels.
// Every launcher enqueues on `stream` and returns the cudaError_t of the launch.
#pragma once

#include <cuda_runtime.h>
#include <stdint.h>

#include "pa.h"

namespace pa {

cudaError_t launch_cache_write(const pa_kv_desc &d, const void *k, const void *v, void *k_cache,
                               void *v_cache, const int64_t *slot_mapping, int32_t num_tokens,
                               cudaStream_t stream);

cudaError_t launch_merge(float *out, float *lse_out, const float *part_o, const float *part_lse,
                         const int32_t *num_parts, int32_t num_seqs, int32_t num_heads,
                         int32_t max_parts, int32_t head_dim, cudaStream_t stream);

// Decode: which kernel variant runs and how many persistent CTAs it uses.
struct DecodePlan {
  int impl;        // PA_DECODE_SIMT or PA_DECODE_MMA
  int slot_heads;  // query heads per partial-result slot of the kernel
  int num_groups;  // kv head groups per sequence (segments per sequence)
  int num_ctas;    // persistent grid size
  size_t workspace_bytes;
};

// Fills `plan` for the descriptor; returns PA_OK or an error with a message.
pa_status plan_decode(const pa_kv_desc &d, int32_t num_seqs, DecodePlan *plan, const char **why);

// Every host-side check of pa_decode's arguments except the workspace, and
// the launch plan (num_seqs == 0 validates the descriptor only); sets the
// last-error string on failure.  Nothing is enqueued.
pa_status validate_decode(const pa_kv_desc *desc, const float *out, const float *lse, const void *q,
                          const void *k_cache, const void *v_cache, const int32_t *block_tables,
                          int32_t max_blocks_per_seq, const int32_t *context_lens, int32_t num_seqs,
                          int32_t max_context_len, float scale, DecodePlan *plan);

// k_new / v_new (pa_decode_append; NULL for pa_decode): sequence s's token
// at position context_lens[s] - 1, [S][kv heads][D] in the cache's 16-bit
// type, written into the caches by the kernel as it attends (MMA kernel).
cudaError_t launch_decode(const pa_kv_desc &d, const DecodePlan &plan, float *out, float *lse,
                          const void *q, const void *k_cache, const void *v_cache,
                          const int32_t *block_tables, int32_t max_blocks_per_seq,
                          const int32_t *context_lens, int32_t num_seqs, float scale,
                          void *workspace, cudaStream_t stream, const void *k_new = nullptr,
                          const void *v_new = nullptr);

pa_status check_prefill(const pa_kv_desc &d, const char **why);

// Every host-side check of pa_prefill_chunk's arguments (num_seqs == 0 or
// max_q_len == 0 validates the descriptor only); sets the last-error string
// on failure.  Nothing is enqueued.
pa_status validate_prefill(const pa_kv_desc *desc, const float *out, const float *lse, const void *q,
                           const int32_t *query_start_loc, const void *k_cache, const void *v_cache,
                           const int32_t *block_tables, int32_t max_blocks_per_seq, const int32_t *context_lens,
                           int32_t num_seqs, int32_t max_q_len, int32_t max_context_len, float scale);

// The single-launch mixed step (pa_mixed.cu): which descriptors it takes,
// and its launch.  The decode plan sizes the decode partitions and the
// workspace, whose head also holds the launch's work counters.
pa_status check_mixed(const pa_kv_desc &d, const DecodePlan &plan, const char **why);
// The decode part's plan in the single-launch step (more partitions than SMs)
// from pa_decode's plan for the same batch.
DecodePlan mixed_plan(const pa_kv_desc &d, int32_t num_dec_seqs, const DecodePlan &plan);
cudaError_t launch_mixed(const pa_kv_desc &d, const DecodePlan &plan, float *dec_out, float *dec_lse,
                         const void *dec_q, const int32_t *dec_block_tables, int32_t dec_max_blocks,
                         const int32_t *dec_context_lens, int32_t num_dec_seqs, float *pf_out, float *pf_lse,
                         const void *pf_q, const int32_t *query_start_loc, const int32_t *pf_block_tables,
                         int32_t pf_max_blocks, const int32_t *pf_context_lens, int32_t num_pf_seqs, int32_t max_q_len,
                         const void *k_cache, const void *v_cache, float scale, void *workspace,
                         cudaStream_t stream, const void *k_new = nullptr, const void *v_new = nullptr,
                         int64_t num_new_rows = 0);

// prefix_mode: every query of sequence s comes after all context_lens[s]
// keys and sees them all (shared-prefix / cascade attention) instead of the
// causal chunk positions; the keys are cut into num_splits splits of
// split_len (a multiple of 128) and split i writes output slot i of
// out_slots per (row, head).
cudaError_t launch_prefill(const pa_kv_desc &d, float *out, float *lse, const void *q,
                           const int32_t *query_start_loc, const void *k_cache,
                           const void *v_cache, const int32_t *block_tables,
                           int32_t max_blocks_per_seq, const int32_t *context_lens,
                           int32_t num_seqs, int32_t max_q_len, float scale, cudaStream_t stream,
                           bool prefix_mode = false, int num_splits = 1, int split_len = 0, int out_slots = 1);

// tcgen05 (tensor-memory) prefill kernel for bf16 and fp16 caches; pair_p:
// P as a hi + lo pair of the cache's type instead of one fp16 value.
cudaError_t launch_prefill_tc(const pa_kv_desc &d, float *out, float *lse, const void *q,
                              const int32_t *query_start_loc, const void *k_cache, const void *v_cache,
                              const int32_t *block_tables, int32_t max_blocks_per_seq, const int32_t *context_lens,
                              int32_t num_seqs, int32_t max_q_len, float scale, cudaStream_t stream,
                              bool prefix_mode, int num_splits, int split_len, int out_slots, bool pair_p);

// The prefill kernel a descriptor selects (a pa_prefill_impl value other
// than AUTO).
int prefill_impl_of(const pa_kv_desc &d);

// The balanced tcgen05 prefill (pa_prefill_chunk_balanced): one CTA per SM,
// the KV iterations of all (query tile, kv head) items dealt out evenly, an
// item cut between CTAs merged in the launch.  It takes batches of at most
// kPrefillSkMaxPairs (sequence, query tile) pairs with a tcgen05 prefill
// kernel selected; others run the plain grid.  Workspace bytes (zero-filled
// once before the first use) and the launch.
constexpr long long kPrefillSkMaxPairs = 16384;
size_t prefill_sk_workspace_bytes(const pa_kv_desc &d, int32_t num_seqs, int32_t max_q_len);
bool prefill_sk_applies(const pa_kv_desc &d, int32_t num_seqs, int32_t max_q_len);
// ... and whether its unit count (KV iterations of all items) stays below 2^31
bool prefill_sk_units_fit(const pa_kv_desc &d, int32_t num_seqs, int32_t max_q_len, int32_t max_blocks_per_seq);
// Whether the balanced kernel is expected to beat the grid: fewer items than
// SMs, with contexts long enough that the SMs the grid leaves idle cost more
// than the pieces' partial outputs and merges.
bool prefill_sk_pays(const pa_kv_desc &d, int32_t num_seqs, int32_t max_q_len, int32_t max_context_len);
// pa_prefill_chunk_balanced's choice: the balanced kernel (true) or the grid
bool prefill_balanced_chosen(const pa_kv_desc &d, int32_t num_seqs, int32_t max_q_len, int32_t max_context_len,
                             int32_t max_blocks_per_seq);
cudaError_t launch_prefill_tc_sk(const pa_kv_desc &d, float *out, float *lse, const void *q,
                                 const int32_t *query_start_loc, const void *k_cache, const void *v_cache,
                                 const int32_t *block_tables, int32_t max_blocks_per_seq,
                                 const int32_t *context_lens, int32_t num_seqs, int32_t max_q_len, float scale,
                                 void *workspace, cudaStream_t stream);

// Copy-on-write of whole blocks (all kv heads) of both caches.
cudaError_t launch_copy_blocks(const pa_kv_desc &d, void *k_cache, void *v_cache, const int32_t *src_blocks,
                               const int32_t *dst_blocks, int32_t num_pairs, cudaStream_t stream);

// Prefix-cache page bookkeeping (bind a hit's pages, release owners).
cudaError_t launch_bind_blocks(const pa_kv_desc &d, int32_t *block_tables, int32_t max_blocks_per_seq,
                               int32_t num_rows, const int32_t *seq_rows, const int32_t *hit_start,
                               const int32_t *hit_blocks, int32_t num_seqs, int32_t *refcounts, cudaStream_t stream);
cudaError_t launch_release_blocks(const pa_kv_desc &d, int32_t *block_tables, int32_t max_blocks_per_seq,
                                  int32_t num_rows, const int32_t *seq_rows, const int32_t *block_counts,
                                  int32_t num_seqs, int32_t *refcounts, int32_t *free_list, int32_t *free_count,
                                  cudaStream_t stream);

// Number of SMs of the current device (cached per device).
int device_sm_count();

// Test hook (pa_test_stall_pipelines): while `stall` is set, the decode and
// tcgen05 prefill kernels launched issue no copies, so that their bounded
// waits run out; every bounded wait of every launch gives up after wait_ns.
constexpr unsigned long long kDefaultWaitNs = 2000000000ull;  // 2 s
struct TestHooks {
  int stall;
  unsigned long long wait_ns;
};
TestHooks test_hooks();

// Sets the message pa_last_error() returns on this thread.
void set_last_error(const char *msg);

}  // namespace pa
