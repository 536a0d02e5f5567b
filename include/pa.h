/*
 * pa.h -- C ABI of a paged KV attention library for one NVIDIA GB300 (sm_103a).
 *
 * The operation is attention over a block-paged KV cache for a continuous
 * batch of variable-length sequences, the "paged attention (block-paged KV
 * cache)" and "chunked prefill" of the vllm.cpp engine ("What's implemented
 * (CPU, behaviorally tested)", Engine core and Model forward bullets, of the
 * vllm.cpp repository page) with its "Block-Paged KV Cache (FP8/FP16)" (the
 * "vllm.cpp ARCHITECTURE OVERVIEW" figure of "Building and Deploying vllm.cpp
 * ...") and block size 16 ("Step 4: Serving Qwen", --block-size 16).
 *
 * Interface conventions follow the pages' own C ABI ("Library API (C ABI)" of
 * the vllm.cpp README): flat, exception-free, versioned with a runtime version
 * query, grows only by appending struct fields whose zero value keeps the old
 * behaviour, and reports failure as a status code plus a last-error string.
 *
 * Memory layout (the pages name no layout; this one is the library's choice):
 *   k_cache, v_cache : [num_blocks][num_kv_heads][block_size][head_dim]
 *                      bf16 or fp16, or one E4M3 or E5M2 byte per element for
 *                      FP8 KV.
 *   q (decode)       : [num_seqs][num_q_heads][head_dim] bf16 (fp16 with an
 *                      fp16 cache)
 *   q (prefill)      : [total_query_tokens][num_q_heads][head_dim], same type
 *   out              : same shape as q, fp32
 *   lse (optional)   : [rows][num_q_heads] fp32, natural-log log-sum-exp of
 *                      the scaled scores of each output row
 *   block_tables     : int32 [num_seqs][max_blocks_per_seq], physical block
 *                      id of each logical block of each sequence
 *   context_lens     : int32 [num_seqs], KV tokens of each sequence including
 *                      the ones written this step
 *   slot_mapping     : int64 [num_tokens], slot = block * block_size + offset;
 *                      a negative slot means "skip this token"
 * Query head h attends kv head h / (num_q_heads / num_kv_heads).
 *
 * Ownership: every pointer is caller-owned device memory unless its comment
 * says "host".  One exception: out and lse of pa_decode, pa_decode_append and
 * pa_decode_static may also be pinned host memory (cudaHostAlloc,
 * cudaMallocHost or cudaHostRegister), which unified addressing maps into the
 * device's address space at the same address.  The decode kernels write
 * those arrays with plain stores only, so the step's result goes straight to
 * the host (over NVLink-C2C on a Grace-Blackwell system).  The result is
 * there once the stream has completed the call.  The library allocates no device memory and keeps no state
 * between calls apart from the thread-local error string and a per-device
 * cache of launch limits (SM count, occupancy).
 *
 * Asynchrony: every compute entry point enqueues work on `stream` (a
 * cudaStream_t; NULL = the legacy default stream) and returns without
 * synchronising.  PA_OK means "validated and enqueued".  Argument errors are
 * detected on the host before anything is enqueued; a CUDA launch error is
 * reported as PA_ERR_CUDA.
 *
 * Device-array contents (block ids, lengths, slots) are the caller's
 * contract.  With pa_kv_desc.check_indices == 0 (the default) they are not
 * checked on the device: a block id outside [0, num_blocks), a context
 * length outside [0, max_blocks_per_seq * block_size], or a slot outside the
 * pool reads or writes out of bounds.  With check_indices == 1 every such
 * value is range-checked on the device before it is used; a value out of
 * range sets PA_DEVERR_BAD_INDEX in the error words, and the access is
 * redirected into the cache (a block id becomes block 0, a length is clamped
 * into its range) or skipped (a cache-write slot, a block copy), so that no
 * access leaves the buffers.  The results of a call that reported
 * PA_DEVERR_BAD_INDEX are meaningless.
 *
 * Failures on the device: every wait of a kernel on its own pipeline (a copy
 * landing, a tensor-core product finishing) is bounded by a 2 s limit.  A
 * kernel whose wait runs out sets PA_DEVERR_WAIT_TIMEOUT in its error words,
 * waits (bounded) for its own copies and products in flight, frees what it
 * holds and returns; its outputs are then incomplete.  The error words are
 * the caller's pa_kv_desc.error_word (every kernel, when given) and, for
 * pa_decode and pa_prefill_chunk_balanced, the first int32 of the
 * workspace.  Kernels never trap.
 */
#ifndef PA_H_
#define PA_H_

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* 1: pa_kv_desc up to prefill_impl; cache write, decode, prefill, merge.
 * 2: pa_kv_desc gains sliding_window, attention_chunk, k_scales, v_scales
 *    (appended); PA_KV_F16; pa_prefix_attention, pa_copy_blocks.
 * 3: pa_kv_desc gains error_word, check_indices (appended); PA_DEVERR_*;
 *    PA_PREFILL_TCGEN05_PAIR; pa_test_stall_pipelines, pa_bind_blocks,
 *    pa_release_blocks, pa_mixed_workspace_size, pa_mixed_attention.
 * 4: pa_prefill_workspace_size, pa_prefill_chunk_balanced,
 *    pa_prefill_balanced_chosen, pa_test_prefill_schedule, pa_decode_append,
 *    pa_mixed_attention_append. */
#define PA_ABI_VERSION 4

/* Symbols of the shared library; everything else in it stays hidden. */
#if defined(__GNUC__)
#define PA_API __attribute__((visibility("default")))
#else
#define PA_API
#endif

struct CUstream_st; /* cudaStream_t is `struct CUstream_st *` */
typedef struct CUstream_st *pa_stream_t;

typedef enum {
  PA_OK = 0,
  PA_ERR_INVALID_ARG = 1, /* null/misaligned pointer, bad size or shape      */
  PA_ERR_UNSUPPORTED = 2, /* valid but not implemented (e.g. head_dim 96)   */
  PA_ERR_WORKSPACE = 3,   /* workspace missing or smaller than required     */
  PA_ERR_CUDA = 4         /* a CUDA runtime call or launch failed           */
} pa_status;

typedef enum {
  PA_KV_BF16 = 0,     /* bf16 K/V, bit copies of the written values          */
  PA_KV_FP8_E4M3 = 1, /* OCP E4M3 bytes, fp32 scales per tensor or kv head */
  PA_KV_FP8_E5M2 = 2, /* OCP E5M2 bytes, fp32 scales per tensor or kv head */
  PA_KV_F16 = 3       /* fp16 K/V of an fp16 model: q and the written rows
                         are fp16 too; bit copies ("Block-Paged KV Cache
                         (FP8/FP16)")                                      */
} pa_kv_dtype;

/* Bits the kernels OR into an error word (see "Failures on the device"). */
#define PA_DEVERR_WAIT_TIMEOUT 1 /* a bounded wait ran out; outputs incomplete */
#define PA_DEVERR_BAD_INDEX 2    /* check_indices: a block id, length or slot
                                    was out of range; results meaningless      */
#define PA_DEVERR_FP16_RANGE 4   /* the tcgen05 prefill (PA_PREFILL_TCGEN05) met a
                                    finite bf16 V value (or, with an 8-bit
                                    cache, a bf16 q value) of magnitude >=
                                    65536, beyond its fp16 products; the rows
                                    using it are wrong: use
                                    PA_PREFILL_TCGEN05_PAIR (V) or
                                    PA_PREFILL_MMA_SYNC                       */
#define PA_DEVERR_REFCOUNT 8     /* pa_release_blocks met a page with no owner
                                    left; that entry was left untouched        */

/* Which decode kernel pa_decode runs.  0 lets the library choose. */
typedef enum {
  PA_DECODE_AUTO = 0,
  PA_DECODE_SIMT = 1,  /* CUDA-core dot products, group size <= 4          */
  PA_DECODE_MMA = 2    /* tensor-core (mma.sync) tiles, any group size <= 16 */
} pa_decode_impl;

/* Which prefill kernel pa_prefill_chunk runs.  0 lets the library choose. */
typedef enum {
  PA_PREFILL_AUTO = 0,
  PA_PREFILL_MMA_SYNC = 1,    /* warp-level mma.sync tiles; every cache type; P
                                 as a hi + lo pair                              */
  PA_PREFILL_TCGEN05 = 2,     /* tcgen05 tensor-memory tiles; bf16 and fp16
                                 caches, and 8-bit caches with head_dim 128
                                 (widened to fp16 in shared memory, q staged
                                 in fp16); P.V in fp16 (see
                                 PA_DEVERR_FP16_RANGE)                          */
  PA_PREFILL_TCGEN05_PAIR = 3 /* tcgen05 tiles with P as a hi + lo pair of the
                                 cache's type: any bf16 range, more tensor
                                 work; bf16 and fp16 caches                     */
} pa_prefill_impl;

/*
 * Shape of the KV pool.  Zero-initialise, then set the fields.  Fields are
 * only ever appended; a zero in an appended field keeps earlier behaviour.
 *   block_size   : tokens per block; 16 is the only supported value.
 *   head_dim     : 64 or 128.
 *   num_q_heads  : a multiple of num_kv_heads; group size g = q / kv <= 16.
 *   k_scale, v_scale : FP8 only.  Cached value = stored E4M3 / E5M2 value *
 *                  scale.
 *                  0 means 1.0.  Ignored for bf16 and fp16.
 *   decode_impl  : a pa_decode_impl value.
 *   prefill_impl : a pa_prefill_impl value.
 *   sliding_window, attention_chunk : local attention ("Local-attention KV +
 *                  sliding-window operator -- SlidingWindowSpec and
 *                  ChunkedLocalAttentionSpec" of the vllm.cpp repository
 *                  listing).  A query at position p attends keys from
 *                  p - sliding_window + 1 (a window of sliding_window keys
 *                  ending at p) and from (p / attention_chunk) *
 *                  attention_chunk (its own chunk) up to p; 0 disables either,
 *                  with both the later start applies.  Applies to pa_decode,
 *                  pa_decode_static and pa_prefill_chunk; must be >= 0.
 *   k_scales, v_scales : FP8 only, optional.  Device arrays of num_kv_heads
 *                  fp32 scales, one per kv head (per-head scaling of the
 *                  8-bit pages; the pages name E4M3/E5M2 pages but no
 *                  scaling scheme).  Where given, kv head h uses its entry
 *                  instead of k_scale / v_scale in the cache write, decode
 *                  and prefill; NULL keeps the per-tensor scale.  4-byte
 *                  aligned, owned by the caller, read by the kernels at run
 *                  time (so they must stay valid until the work completes).
 *                  Must be NULL for bf16 and fp16 caches.
 *   error_word   : optional device int32, owned by the caller, 4-byte
 *                  aligned.  Every kernel of a call made with this
 *                  descriptor ORs its PA_DEVERR_* bits into it (atomically);
 *                  nothing clears it, so zero it before the calls it should
 *                  watch and read it after they complete.  NULL: no such
 *                  word (pa_decode still reports into its workspace).
 *   check_indices: 0 or 1; 1 range-checks block ids, context lengths,
 *                  query-chunk lengths, cache-write slots and block-copy ids
 *                  on the device (see "Device-array contents" above).
 */
typedef struct {
  int32_t num_blocks;
  int32_t block_size;
  int32_t num_kv_heads;
  int32_t num_q_heads;
  int32_t head_dim;
  int32_t kv_dtype; /* pa_kv_dtype */
  float k_scale;
  float v_scale;
  int32_t decode_impl;     /* pa_decode_impl */
  int32_t prefill_impl;    /* pa_prefill_impl */
  int32_t sliding_window;  /* 0: none */
  int32_t attention_chunk; /* 0: none */
  const float *k_scales;   /* NULL: per-tensor k_scale */
  const float *v_scales;   /* NULL: per-tensor v_scale */
  int32_t *error_word;     /* NULL: none */
  int32_t check_indices;   /* 0: contents unchecked */
} pa_kv_desc;

/* PA_ABI_VERSION of the loaded library. */
PA_API int pa_abi_version(void);

/* Message of the last failing call on this thread ("" if none).  The pointer
 * stays valid until the next library call on the same thread. */
PA_API const char *pa_last_error(void);

/*
 * Slot-mapped cache write.  For every token i < num_tokens with
 * slot_mapping[i] >= 0, block = slot / block_size and offset = slot %
 * block_size; for every kv head h, the cache row (block, h, offset) receives
 * k[i][h][:] (v likewise).  bf16 and fp16 KV store the bits unchanged.  FP8 KV stores
 * e4m3 (or e5m2) of fl32(x) / k_scale, rounded to nearest even, with finite
 * overflow saturating to +-448 (E4M3) or +-57344 (E5M2, where +-inf
 * saturates too), and NaN kept as a NaN code.
 *   k, v : [num_tokens][num_kv_heads][head_dim] bf16 (fp16 for an fp16
 *          cache), 16-byte aligned.
 * The write of a prefix-cache hit must not target a block shared with another
 * sequence ("Zero-Copy Cache Hits" of "1. Technical Mechanics of the Radix
 * Cache" binds sequences to the same physical pages; writing into one would
 * change all of them).  Duplicate slots in one call race.
 * num_tokens == 0 enqueues nothing and returns PA_OK.
 */
PA_API pa_status pa_cache_write(const pa_kv_desc *desc, const void *k, const void *v, void *k_cache,
                         void *v_cache, const int64_t *slot_mapping, int32_t num_tokens,
                         pa_stream_t stream);

/*
 * Bytes of scratch that pa_decode needs for num_seqs sequences on the current
 * device.  Zero-fill the workspace once before its first use; it may then be
 * reused by consecutive calls on one stream (each call that completes without
 * error leaves its error word and its merge counters at zero again; the rest
 * holds the last call's partial results).  Calls that overlap on the GPU need
 * separate workspaces.  After a call completes, the first int32 of the
 * workspace holds the PA_DEVERR_* bits it reported; if it is not zero, the
 * merge counters may be left behind too: zero-fill the whole workspace again
 * before its next use.
 */
PA_API size_t pa_decode_workspace_size(const pa_kv_desc *desc, int32_t num_seqs, int32_t max_context_len);

/*
 * Decode attention, split-KV.  Sequence s has one query q[s] at position
 * context_lens[s] - 1; query head h attends all tokens [0, context_lens[s]) of
 * kv head h / g through block_tables[s]:
 *   out[s][h] = sum_t softmax_t(scale * q[s][h] . K_t) V_t     (fp32)
 *   lse[s][h] = ln sum_t exp(scale * q[s][h] . K_t)          (if lse != NULL)
 * A sequence with context length 0 gets out = 0 and lse = -inf.
 * The KV range of long sequences is split across CTAs and the pieces are
 * merged by log-sum-exp inside the same launch.
 *   max_context_len : an upper bound of context_lens (host value).
 *   workspace       : pa_decode_workspace_size() bytes, zero-filled once.
 */
PA_API pa_status pa_decode(const pa_kv_desc *desc, float *out, float *lse, const void *q,
                    const void *k_cache, const void *v_cache, const int32_t *block_tables,
                    int32_t max_blocks_per_seq, const int32_t *context_lens, int32_t num_seqs,
                    int32_t max_context_len, float scale, void *workspace, size_t workspace_bytes,
                    pa_stream_t stream);

/*
 * Chunked-prefill causal attention over the paged cache.  Sequence s owns the
 * packed query rows [query_start_loc[s], query_start_loc[s+1]); with q_len
 * their count, query i of it sits at position context_lens[s] - q_len + i and
 * attends keys [0, position] of its kv head (the chunk's own K/V must have
 * been written by pa_cache_write first).  Blocks shared by several tables
 * (a prefix-cache hit) are only read.
 *   q   : [query_start_loc[num_seqs]][num_q_heads][head_dim] bf16 (fp16 for
 *         an fp16 cache)
 *   out : same shape, fp32; lse (optional) [rows][num_q_heads]
 *   query_start_loc : int32 [num_seqs + 1], non-decreasing, starting at 0,
 *                     q_len <= context_lens[s].
 *   max_q_len : an upper bound of the q_len values (host value).
 * num_seqs is at most 65535 per call (PA_ERR_UNSUPPORTED above).
 */
PA_API pa_status pa_prefill_chunk(const pa_kv_desc *desc, float *out, float *lse, const void *q,
                           const int32_t *query_start_loc, const void *k_cache,
                           const void *v_cache, const int32_t *block_tables,
                           int32_t max_blocks_per_seq, const int32_t *context_lens,
                           int32_t num_seqs, int32_t max_q_len, int32_t max_context_len,
                           float scale, pa_stream_t stream);

/*
 * A decode step's cache write and decode attention in one launch: the decode
 * half of one pass of the engine loop (the "C++20 Continuous Batching Loop"
 * figure of "Building and Deploying vllm.cpp ...": the new token's K/V go into
 * the paged cache, then attention reads the sequence's whole context).
 * Sequence s appends one token at position context_lens[s] - 1 (context_lens
 * already count it), whose K and V rows are k_new[s] and v_new[s]: the call writes
 * them into the caches at that position through block_tables (what
 * pa_cache_write does for those slots) and computes pa_decode's output over
 * all context_lens[s] tokens, the appended one included.  The kernel puts
 * the new rows into the tiles it stages as it reads each sequence's last
 * block, so the attention does not wait for a separate write.
 *   k_new, v_new : [num_seqs][num_kv_heads][head_dim] bf16 (fp16 for an fp16
 *                  cache), 16-byte aligned; a sequence with context length 0
 *                  appends nothing.  An 8-bit cache receives the rows encoded
 *                  exactly as pa_cache_write encodes them (same bytes).
 *   the other arguments are pa_decode's (workspace: pa_decode_workspace_size).
 * Runs on the tensor-core decode kernel, for every cache type
 * (PA_ERR_UNSUPPORTED with decode_impl PA_DECODE_SIMT: call pa_cache_write
 * and pa_decode).  Errors found on the host (pa_decode's, NULL or misaligned
 * k_new / v_new: PA_ERR_INVALID_ARG; PA_ERR_UNSUPPORTED; PA_ERR_WORKSPACE)
 * return before anything is enqueued.  With check_indices, an out-of-range block id of a
 * last block is reported and its row is not written.  Two sequences whose
 * last tokens share a slot race, as duplicate slots of pa_cache_write do.
 */
PA_API pa_status pa_decode_append(const pa_kv_desc *desc, float *out, float *lse, const void *q, const void *k_new,
                                  const void *v_new, void *k_cache, void *v_cache, const int32_t *block_tables,
                                  int32_t max_blocks_per_seq, const int32_t *context_lens, int32_t num_seqs,
                                  int32_t max_context_len, float scale, void *workspace, size_t workspace_bytes,
                                  pa_stream_t stream);

/*
 * Bytes of scratch that pa_prefill_chunk_balanced needs for num_seqs chunks
 * of at most max_q_len queries on the current device (0 if the descriptor is
 * invalid).  Same rules as pa_decode's workspace: zero-fill it once before
 * its first use; consecutive calls on one stream may reuse it (a call that
 * completes without error leaves its error word and its piece counters at
 * zero); calls that overlap on the GPU need separate workspaces.  After a
 * call completes, its first int32 holds the PA_DEVERR_* bits the balanced
 * kernel reported; if it is not zero, zero-fill the whole workspace again
 * before its next use.
 */
PA_API size_t pa_prefill_workspace_size(const pa_kv_desc *desc, int32_t num_seqs, int32_t max_q_len);

/*
 * pa_prefill_chunk, with the work spread evenly over the SMs where that pays.
 * Same arguments, same result up to fp32 rounding (within the library's
 * tolerances of pa_prefill_chunk).  pa_prefill_chunk gives every (query tile
 * of 256 / g queries, kv head) item its own CTA, so a batch of n items runs
 * in ceil(n / SMs) waves, and a batch of fewer items than SMs (a few long
 * chunks) leaves SMs idle for the whole launch.  The balanced kernel runs one
 * CTA per SM, each taking an equal share of all items' 128-key tiles; an
 * item whose tiles fall to several CTAs is computed in pieces (the "chunked
 * prefill" chunk cut along its keys), and the last piece to finish merges
 * them by log-sum-exp, as pa_merge_partials does, inside the same launch.
 * It runs when the descriptor selects a tcgen05 prefill kernel, num_seqs *
 * ceil(max_q_len * g / 256) <= 16384, the batch has fewer items than SMs and
 * ceil(max_context_len / 128) * (SMs - items) > 12 * SMs (the SMs the grid
 * would leave idle outweigh the pieces' merges); other batches run
 * pa_prefill_chunk's grid (pa_test_prefill_schedule overrides the choice).
 *   workspace : pa_prefill_workspace_size(desc, num_seqs, max_q_len) bytes,
 *               16-byte aligned, zero-filled before its first use.
 */
/*
 * Which kernel pa_prefill_chunk_balanced runs for a batch of num_seqs chunks
 * of at most max_q_len queries over contexts of at most max_context_len
 * tokens (tables of max_blocks_per_seq blocks): 1 the balanced kernel, 0
 * pa_prefill_chunk's grid, -1 for an invalid descriptor or arguments.  A
 * caller that schedules a step can use it to keep such a prefill out of a
 * single-launch step (see pa_mixed_attention).  Host only; enqueues nothing.
 */
PA_API int32_t pa_prefill_balanced_chosen(const pa_kv_desc *desc, int32_t num_seqs, int32_t max_q_len,
                                          int32_t max_context_len, int32_t max_blocks_per_seq);

PA_API pa_status pa_prefill_chunk_balanced(const pa_kv_desc *desc, float *out, float *lse, const void *q,
                                           const int32_t *query_start_loc, const void *k_cache,
                                           const void *v_cache, const int32_t *block_tables,
                                           int32_t max_blocks_per_seq, const int32_t *context_lens,
                                           int32_t num_seqs, int32_t max_q_len, int32_t max_context_len,
                                           float scale, void *workspace, size_t workspace_bytes,
                                           pa_stream_t stream);

/*
 * Decode and chunked-prefill attention of one continuous-batch step in a
 * single launch (the step of the "C++20 Continuous Batching Loop" in the
 * "vllm.cpp ARCHITECTURE OVERVIEW" figure; the unified scheduler with
 * chunked prefill of the vllm.cpp repository's Engine core bullet).  It
 * computes what pa_decode computes for the dec_* arguments and what
 * pa_prefill_chunk computes for the pf_* arguments, over the same caches,
 * in one persistent launch whose CTAs take the prefill's tiles (longest key
 * ranges first) and then the decode's partitions from one work list: the
 * decode fills the SMs the prefill's last wave leaves idle.  Issue the
 * step's pa_cache_write first, on the same stream (or use
 * pa_mixed_attention_append, which writes the rows in the same launch).
 *   workspace : pa_mixed_workspace_size(desc, num_dec_seqs,
 *               dec_max_context_len) bytes, zero-filled before its first use;
 *               every call that completes without error leaves it ready for
 *               the next (its counters back at zero).  Calls that overlap on
 *               the GPU need separate workspaces.
 * Either part may be empty (num_dec_seqs == 0 or num_pf_seqs == 0).  Takes
 * bf16 and fp16 caches with head_dim 128, decode_impl AUTO or MMA and
 * prefill_impl AUTO or TCGEN05; PA_ERR_UNSUPPORTED otherwise (make the two
 * calls instead).
 */
/* Bytes of scratch pa_mixed_attention needs for num_dec_seqs decode
 * sequences on the current device (0 if the descriptor is invalid). */
PA_API size_t pa_mixed_workspace_size(const pa_kv_desc *desc, int32_t num_dec_seqs, int32_t dec_max_context_len);

PA_API pa_status pa_mixed_attention(const pa_kv_desc *desc, float *dec_out, float *dec_lse, const void *dec_q,
                                    const int32_t *dec_block_tables, int32_t dec_max_blocks_per_seq,
                                    const int32_t *dec_context_lens, int32_t num_dec_seqs,
                                    int32_t dec_max_context_len, float *pf_out, float *pf_lse, const void *pf_q,
                                    const int32_t *query_start_loc, const int32_t *pf_block_tables,
                                    int32_t pf_max_blocks_per_seq, const int32_t *pf_context_lens,
                                    int32_t num_pf_seqs, int32_t max_q_len, int32_t pf_max_context_len,
                                    const void *k_cache, const void *v_cache, float scale, void *workspace,
                                    size_t workspace_bytes, pa_stream_t stream);

/*
 * The whole continuous-batch step in one launch: the step's cache write
 * (what pa_cache_write does for its new tokens) folded into
 * pa_mixed_attention, whose results it computes over the caches with the
 * new tokens in them.  No barrier is needed inside the launch:
 *   - a decode sequence's new row is written, and used, by the warp that
 *     owns the sequence's last block (as in pa_decode_append);
 *   - a prefill chunk's own keys are read from k_new / v_new instead of the
 *     caches, and each tile writes its own queries' rows into the caches.
 *   k_new, v_new : [num_new_rows][num_kv_heads][head_dim] in the cache's
 *                  16-bit type, 16-byte aligned.  Row s < num_dec_seqs is
 *                  decode sequence s's new token (position
 *                  dec_context_lens[s] - 1); row num_dec_seqs +
 *                  query_start_loc[s] + i is prefill sequence s's token i
 *                  (position pf_context_lens[s] - q_len_s + i).
 *   num_new_rows : rows of k_new / v_new (num_dec_seqs +
 *                  query_start_loc[num_pf_seqs]), host value.  With a
 *                  prefill part it must exceed num_dec_seqs; a chunk row
 *                  past it is neither read nor written (PA_DEVERR_BAD_INDEX).
 * Every prefill chunk must start at a multiple of block_size
 * (pf_context_lens[s] - q_len_s), so that a block holds either cached or new
 * tokens.  A chunk that does not is reported on the device
 * (PA_DEVERR_BAD_INDEX) and its outputs are meaningless; for such a step
 * make the pa_cache_write and pa_mixed_attention calls.  The other
 * arguments, restrictions and errors are pa_mixed_attention's; k_new /
 * v_new problems give PA_ERR_INVALID_ARG before anything is enqueued.  Do
 * not issue pa_cache_write for these rows as well.
 */
PA_API pa_status pa_mixed_attention_append(const pa_kv_desc *desc, float *dec_out, float *dec_lse,
                                           const void *dec_q, const int32_t *dec_block_tables,
                                           int32_t dec_max_blocks_per_seq, const int32_t *dec_context_lens,
                                           int32_t num_dec_seqs, int32_t dec_max_context_len, float *pf_out,
                                           float *pf_lse, const void *pf_q, const int32_t *query_start_loc,
                                           const int32_t *pf_block_tables, int32_t pf_max_blocks_per_seq,
                                           const int32_t *pf_context_lens, int32_t num_pf_seqs, int32_t max_q_len,
                                           int32_t pf_max_context_len, const void *k_new, const void *v_new,
                                           int64_t num_new_rows, void *k_cache, void *v_cache, float scale,
                                           void *workspace, size_t workspace_bytes, pa_stream_t stream);

/*
 * Shared-prefix (cascade) attention.  A prefix-cache hit binds several
 * sequences to the same physical pages ("Zero-Copy Cache Hits" of "1.
 * Technical Mechanics of the Radix Cache"); their queries can attend that
 * prefix together, reading it once per kv head instead of once per sequence,
 * and then merge the result with each sequence's own suffix (pa_decode over
 * the suffix's blocks) by pa_merge_partials.  Group j owns the packed query
 * rows [query_start_loc[j], query_start_loc[j+1]) and the prefix of
 * prefix_lens[j] tokens behind prefix_tables[j]; every query of the group
 * attends all of it (no causal mask: the queries come after the prefix).
 * The prefix keys are cut into num_splits splits of c tokens each, c =
 * ceil(max_prefix_len / num_splits) rounded up to a multiple of 128; split i
 * covers keys [i c, min(prefix_len, (i + 1) c)) and is computed by its own
 * CTAs, so that a few long prefixes still fill the GPU.  Split i of row r,
 * head h is written to slot i of out_slots:
 *   q   : [query_start_loc[num_groups]][num_q_heads][head_dim] (q's type as in
 *         pa_prefill_chunk)
 *   out : [rows][num_q_heads][out_slots][head_dim] fp32, each split's result
 *         normalised by its own sum; lse : [rows][num_q_heads][out_slots]
 *         fp32, natural log, required.  A split without keys (an empty or
 *         short prefix) gets out = 0 and lse = -inf, which drop out of the
 *         merge.  Slots >= num_splits are left untouched, so out / lse can be
 *         pa_merge_partials' part_o / part_lse with the suffix in the last slot.
 *   num_splits : >= 1; out_slots : >= num_splits, or 0 for num_splits.
 *   prefix_tables : int32 [num_groups][max_blocks_per_prefix]
 *   prefix_lens   : int32 [num_groups]; max_prefix_len bounds them (host).
 * Local attention does not apply (sliding_window and attention_chunk must be
 * 0).  The kernel is the one pa_prefill_chunk would run for the descriptor.
 */
PA_API pa_status pa_prefix_attention(const pa_kv_desc *desc, float *out, float *lse, const void *q,
                                     const int32_t *query_start_loc, const void *k_cache, const void *v_cache,
                                     const int32_t *prefix_tables, int32_t max_blocks_per_prefix,
                                     const int32_t *prefix_lens, int32_t num_groups, int32_t max_q_len,
                                     int32_t max_prefix_len, int32_t num_splits, int32_t out_slots, float scale,
                                     pa_stream_t stream);

/*
 * Copy-on-write of whole pages: for every i < num_pairs, block dst_blocks[i]
 * of both caches receives the contents of block src_blocks[i] (every kv head
 * and slot), so that a sequence about to write into a page it shares with
 * other sequences (the partly filled last page of a prefix-cache hit) gets a
 * private copy first.
 *   src_blocks, dst_blocks : int32 [num_pairs] device arrays of block ids in
 *                            [0, num_blocks); no dst may repeat or appear
 *                            among the srcs (copies of one call race).
 * num_pairs == 0 enqueues nothing and returns PA_OK.
 */
PA_API pa_status pa_copy_blocks(const pa_kv_desc *desc, void *k_cache, void *v_cache, const int32_t *src_blocks,
                                const int32_t *dst_blocks, int32_t num_pairs, pa_stream_t stream);

/*
 * Prefix-cache page bookkeeping on the device ("1. Technical Mechanics of
 * the Radix Cache": a hit binds the new sequence's block table directly to
 * the pages of its matched prefix, "Zero-Copy Cache Hits"; eviction returns
 * pages to the global page pool, "LRU Eviction").  The radix tree, the LRU
 * order and the choice of what to evict stay with the caller; these calls
 * keep the page tables and the owner counts on the device.
 *   block_tables : int32 [num_table_rows][max_blocks_per_seq]
 *   refcounts    : int32 [desc->num_blocks], owners of each page
 * Table rows, hit lengths and page ids are always range-checked: an entry
 * outside the table or the pool is skipped and sets PA_DEVERR_BAD_INDEX in
 * desc->error_word (when given).  Owner counts change atomically, so
 * several sequences of one call may share pages; two entries of one call
 * must not write the same table slot.
 *
 * pa_bind_blocks: for every i < num_seqs, table row seq_rows[i] gets the
 * hit's pages hit_blocks[hit_start[i] .. hit_start[i+1]) in its first
 * entries, and each of those pages gains one owner.
 *   seq_rows   : int32 [num_seqs]
 *   hit_start  : int32 [num_seqs + 1], non-decreasing
 *   hit_blocks : int32 [hit_start[num_seqs]]
 */
PA_API pa_status pa_bind_blocks(const pa_kv_desc *desc, int32_t *block_tables, int32_t max_blocks_per_seq,
                                int32_t num_table_rows, const int32_t *seq_rows, const int32_t *hit_start,
                                const int32_t *hit_blocks, int32_t num_seqs, int32_t *refcounts,
                                pa_stream_t stream);

/*
 * pa_release_blocks: for every i < num_seqs, each of the first
 * block_counts[i] pages of table row seq_rows[i] loses one owner and its
 * entry becomes -1 (a finished sequence releases its own row; an evicted
 * cache entry can pass its pages as a row of its own table).  A page whose
 * owner count reaches zero returns to the pool: it is written to
 * free_list[*free_count] and *free_count grows by one (atomically, so the
 * order of the pages a call frees is unspecified).  A page with no owner
 * left is not touched and sets PA_DEVERR_REFCOUNT.
 *   block_counts : int32 [num_seqs]
 *   free_list    : int32 [desc->num_blocks]; free_count : one int32, the
 *                  number of entries already in it (device)
 */
PA_API pa_status pa_release_blocks(const pa_kv_desc *desc, int32_t *block_tables, int32_t max_blocks_per_seq,
                                   int32_t num_table_rows, const int32_t *seq_rows, const int32_t *block_counts,
                                   int32_t num_seqs, int32_t *refcounts, int32_t *free_list, int32_t *free_count,
                                   pa_stream_t stream);

/*
 * Merge of attention results over disjoint key ranges (split-KV pieces, or a
 * shared prefix and a private suffix), by log-sum-exp weighting:
 *   M = max_p lse_p,  w_p = exp(lse_p - M),
 *   out = sum_p w_p o_p / sum_p w_p,  lse_out = M + ln sum_p w_p.
 * Parts with lse = -inf hold no keys and drop out; if all are empty the result
 * is out = 0, lse_out = -inf.
 *   part_o   : [num_seqs][num_heads][max_parts][head_dim] fp32 (each o_p
 *              already normalised by its own softmax sum)
 *   part_lse : [num_seqs][num_heads][max_parts] fp32, natural log
 *   num_parts: int32 [num_seqs] parts used by each sequence (each <=
 *              max_parts), or NULL for max_parts everywhere.
 *   out      : [num_seqs][num_heads][head_dim] fp32; lse_out optional.
 *   head_dim : a multiple of 4, at most 512.
 */
PA_API pa_status pa_merge_partials(float *out, float *lse_out, const float *part_o,
                            const float *part_lse, const int32_t *num_parts, int32_t num_seqs,
                            int32_t num_heads, int32_t max_parts, int32_t head_dim,
                            pa_stream_t stream);

/*
 * Decode without a workspace argument (the paper has no counterpart; this is
 * a convenience of this library).  Same operation, arguments and results as
 * pa_decode, for callers that cannot allocate device memory where they
 * decode: serving loops held to a fixed device-memory budget once the KV
 * pool is sized, runtimes whose device memory is fully planned up front, and
 * plug-ins whose host framework owns the allocator.  The scratch is a fixed 8 MiB array in the library's own device
 * memory (held on every GPU that loads the library until the process exits);
 * a batch needing more scratch than that (pa_decode_workspace_size) is
 * rejected with PA_ERR_WORKSPACE.  The call allocates nothing: it clears the
 * array's error word and merge counters with cudaMemsetAsync on `stream` and
 * enqueues the decode kernels there.  The first call on each device looks up
 * the array's device address (cudaGetSymbolAddress, with that device
 * current); make that first call before any stream capture.  All calls share
 * the one array, so calls that may overlap on the GPU (different streams
 * without ordering between them) race; serialise them, or use pa_decode with
 * separate workspaces.  The array's own error word is cleared by every call,
 * so device failures (PA_DEVERR_*) of pa_decode_static are visible only
 * through desc->error_word: pass one to see them.  Arguments are validated
 * as in pa_decode before anything is enqueued.
 */
PA_API pa_status pa_decode_static(const pa_kv_desc *desc, float *out, float *lse, const void *q,
                                  const void *k_cache, const void *v_cache, const int32_t *block_tables,
                                  int32_t max_blocks_per_seq, const int32_t *context_lens, int32_t num_seqs,
                                  int32_t max_context_len, float scale, pa_stream_t stream);

/*
 * Test hook for the failure path (no counterpart on the pages).  While
 * enabled (enable != 0), the producers of the decode and tcgen05 prefill
 * kernels launched afterwards issue no copies and signal nothing, so the
 * kernels' bounded waits run out: they report PA_DEVERR_WAIT_TIMEOUT, free
 * what they hold and return, with nothing in flight.  wait_limit_ns (> 0)
 * replaces the 2 s limit of every bounded wait while enabled, so a test
 * does not wait long.  Process-wide; pass enable = 0 to restore normal
 * launches.  Never enable it outside tests.
 */
PA_API pa_status pa_test_stall_pipelines(int32_t enable, int64_t wait_limit_ns);

/*
 * Test hook (no counterpart on the pages): which schedule
 * pa_prefill_chunk_balanced runs.  0 (the default): the library's choice; 1:
 * the balanced kernel wherever it applies (a tcgen05 prefill kernel, the
 * batch within its limits); 2: always pa_prefill_chunk's grid.
 * Process-wide; returns PA_ERR_INVALID_ARG for other values.
 */
PA_API pa_status pa_test_prefill_schedule(int32_t schedule);

#ifdef __cplusplus
}
#endif

#endif /* PA_H_ */
