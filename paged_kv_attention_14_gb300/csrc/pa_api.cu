// pa_api.cu -- the extern "C" entry points declared in include/pa.h.
//
// Host-side argument checks (nothing is enqueued when one fails), the
// thread-local error string, workspace sizing and dispatch to the kernels.
// The conventions -- flat, exception-free functions, a status code plus a
// last-error string, a runtime ABI version, structs that only grow by
// appending fields -- follow the pages' own "Library API (C ABI)" section of
// the vllm.cpp README.
#include <stdio.h>
#include <string.h>

#include <atomic>

#include "pa.h"
#include "pa_internal.h"

namespace {

thread_local char g_last_error[512] = "";

pa_status fail(pa_status st, const char *fmt, const char *detail = nullptr) {
  snprintf(g_last_error, sizeof g_last_error, fmt, detail ? detail : "");
  return st;
}

pa_status ok() {
  g_last_error[0] = '\0';
  return PA_OK;
}

bool aligned16(const void *p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

pa_status check_desc(const pa_kv_desc *d) {
  if (!d) return fail(PA_ERR_INVALID_ARG, "desc is NULL%s");
  if (d->block_size != 16) return fail(PA_ERR_UNSUPPORTED, "block_size must be 16%s");
  if (d->head_dim != 64 && d->head_dim != 128)
    return fail(PA_ERR_UNSUPPORTED, "head_dim must be 64 or 128%s");
  if (d->num_kv_heads <= 0 || d->num_q_heads <= 0)
    return fail(PA_ERR_INVALID_ARG, "num_kv_heads and num_q_heads must be positive%s");
  if (d->num_q_heads % d->num_kv_heads != 0)
    return fail(PA_ERR_INVALID_ARG, "num_q_heads must be a multiple of num_kv_heads%s");
  if (d->num_q_heads / d->num_kv_heads > 16)
    return fail(PA_ERR_UNSUPPORTED, "group size num_q_heads / num_kv_heads must be <= 16%s");
  if (d->kv_dtype != PA_KV_BF16 && d->kv_dtype != PA_KV_FP8_E4M3 && d->kv_dtype != PA_KV_FP8_E5M2 &&
      d->kv_dtype != PA_KV_F16)
    return fail(PA_ERR_INVALID_ARG, "kv_dtype must be PA_KV_BF16, PA_KV_F16, PA_KV_FP8_E4M3 or PA_KV_FP8_E5M2%s");
  if (d->num_blocks < 0) return fail(PA_ERR_INVALID_ARG, "num_blocks must be >= 0%s");
  if (d->sliding_window < 0 || d->attention_chunk < 0)
    return fail(PA_ERR_INVALID_ARG, "sliding_window and attention_chunk must be >= 0%s");
  const bool kv8 = d->kv_dtype == PA_KV_FP8_E4M3 || d->kv_dtype == PA_KV_FP8_E5M2;
  if (kv8 && (!(d->k_scale >= 0.f) || !(d->v_scale >= 0.f)))
    return fail(PA_ERR_INVALID_ARG, "k_scale and v_scale must be >= 0 (0 means 1)%s");
  if (!kv8 && (d->k_scales || d->v_scales))
    return fail(PA_ERR_INVALID_ARG, "per-head k_scales / v_scales apply to FP8 caches only%s");
  if ((reinterpret_cast<uintptr_t>(d->k_scales) | reinterpret_cast<uintptr_t>(d->v_scales)) & 3u)
    return fail(PA_ERR_INVALID_ARG, "k_scales and v_scales must be 4-byte aligned%s");
  if (reinterpret_cast<uintptr_t>(d->error_word) & 3u)
    return fail(PA_ERR_INVALID_ARG, "error_word must be 4-byte aligned%s");
  if (d->check_indices != 0 && d->check_indices != 1)
    return fail(PA_ERR_INVALID_ARG, "check_indices must be 0 or 1%s");
  return PA_OK;
}

std::atomic<int> g_test_stall{0};
std::atomic<unsigned long long> g_test_wait_ns{0};
std::atomic<int> g_test_schedule{0};  // pa_test_prefill_schedule

pa_status cuda_fail(cudaError_t e) {
  return fail(PA_ERR_CUDA, "CUDA error: %s", cudaGetErrorString(e));
}

}  // namespace

namespace pa {

void set_last_error(const char *msg) { snprintf(g_last_error, sizeof g_last_error, "%s", msg); }

bool prefill_balanced_chosen(const pa_kv_desc &d, int32_t num_seqs, int32_t max_q_len, int32_t max_context_len,
                             int32_t max_blocks_per_seq) {
  // the balanced kernel where it applies and pays (or as the test hook says)
  const int forced = g_test_schedule.load(std::memory_order_relaxed);
  return prefill_sk_applies(d, num_seqs, max_q_len) && prefill_sk_units_fit(d, num_seqs, max_q_len, max_blocks_per_seq) &&
         (forced == 1 || (forced == 0 && prefill_sk_pays(d, num_seqs, max_q_len, max_context_len)));
}

TestHooks test_hooks() {
  TestHooks h;
  h.stall = g_test_stall.load(std::memory_order_relaxed);
  const unsigned long long w = g_test_wait_ns.load(std::memory_order_relaxed);
  h.wait_ns = (h.stall && w) ? w : kDefaultWaitNs;
  return h;
}

pa_status validate_decode(const pa_kv_desc *desc, const float *out, const float *lse, const void *q,
                          const void *k_cache, const void *v_cache, const int32_t *block_tables,
                          int32_t max_blocks_per_seq, const int32_t *context_lens, int32_t num_seqs,
                          int32_t max_context_len, float scale, DecodePlan *plan) {
  pa_status st = check_desc(desc);
  if (st != PA_OK) return st;
  if (num_seqs < 0) return fail(PA_ERR_INVALID_ARG, "num_seqs must be >= 0%s");
  if (num_seqs == 0) return PA_OK;
  if (!out || !q || !k_cache || !v_cache || !block_tables || !context_lens)
    return fail(PA_ERR_INVALID_ARG,
                "out, q, k_cache, v_cache, block_tables and context_lens must be non-NULL%s");
  if (!aligned16(out) || !aligned16(q) || !aligned16(k_cache) || !aligned16(v_cache))
    return fail(PA_ERR_INVALID_ARG, "out, q, k_cache and v_cache must be 16-byte aligned%s");
  if ((reinterpret_cast<uintptr_t>(block_tables) & 3u) || (reinterpret_cast<uintptr_t>(context_lens) & 3u) ||
      (reinterpret_cast<uintptr_t>(lse) & 3u))
    return fail(PA_ERR_INVALID_ARG, "block_tables, context_lens and lse must be 4-byte aligned%s");
  if (max_blocks_per_seq <= 0) return fail(PA_ERR_INVALID_ARG, "max_blocks_per_seq must be positive%s");
  if (max_context_len < 0 || static_cast<int64_t>(max_context_len) > static_cast<int64_t>(max_blocks_per_seq) * 16)
    return fail(PA_ERR_INVALID_ARG, "max_context_len must lie in [0, max_blocks_per_seq * block_size]%s");
  if (!(scale == scale)) return fail(PA_ERR_INVALID_ARG, "scale is NaN%s");
  const char *why = "";
  st = plan_decode(*desc, num_seqs, plan, &why);
  if (st != PA_OK) return fail(st, "%s", why);
  return PA_OK;
}

pa_status validate_prefill(const pa_kv_desc *desc, const float *out, const float *lse, const void *q,
                           const int32_t *query_start_loc, const void *k_cache, const void *v_cache,
                           const int32_t *block_tables, int32_t max_blocks_per_seq, const int32_t *context_lens,
                           int32_t num_seqs, int32_t max_q_len, int32_t max_context_len, float scale) {
  pa_status st = check_desc(desc);
  if (st != PA_OK) return st;
  if (num_seqs < 0 || max_q_len < 0) return fail(PA_ERR_INVALID_ARG, "num_seqs and max_q_len must be >= 0%s");
  if (num_seqs == 0 || max_q_len == 0) return PA_OK;
  if (num_seqs > 65535)  // one grid row of CTAs per sequence
    return fail(PA_ERR_UNSUPPORTED, "a prefill takes at most 65535 sequences per call%s");
  if (!out || !q || !query_start_loc || !k_cache || !v_cache || !block_tables || !context_lens)
    return fail(PA_ERR_INVALID_ARG,
                "out, q, query_start_loc, k_cache, v_cache, block_tables and context_lens must be non-NULL%s");
  if (!aligned16(out) || !aligned16(q) || !aligned16(k_cache) || !aligned16(v_cache))
    return fail(PA_ERR_INVALID_ARG, "out, q, k_cache and v_cache must be 16-byte aligned%s");
  if ((reinterpret_cast<uintptr_t>(block_tables) & 3u) || (reinterpret_cast<uintptr_t>(context_lens) & 3u) ||
      (reinterpret_cast<uintptr_t>(query_start_loc) & 3u) || (reinterpret_cast<uintptr_t>(lse) & 3u))
    return fail(PA_ERR_INVALID_ARG,
                "block_tables, context_lens, query_start_loc and lse must be 4-byte aligned%s");
  if (max_blocks_per_seq <= 0) return fail(PA_ERR_INVALID_ARG, "max_blocks_per_seq must be positive%s");
  if (max_context_len < 0 || static_cast<int64_t>(max_context_len) > static_cast<int64_t>(max_blocks_per_seq) * 16)
    return fail(PA_ERR_INVALID_ARG, "max_context_len must lie in [0, max_blocks_per_seq * block_size]%s");
  if (!(scale == scale)) return fail(PA_ERR_INVALID_ARG, "scale is NaN%s");
  const char *why = "";
  st = check_prefill(*desc, &why);
  if (st != PA_OK) return fail(st, "%s", why);
  return PA_OK;
}

}  // namespace pa

extern "C" {

int pa_abi_version(void) { return PA_ABI_VERSION; }

const char *pa_last_error(void) { return g_last_error; }

pa_status pa_cache_write(const pa_kv_desc *desc, const void *k, const void *v, void *k_cache,
                         void *v_cache, const int64_t *slot_mapping, int32_t num_tokens,
                         pa_stream_t stream) {
  pa_status st = check_desc(desc);
  if (st != PA_OK) return st;
  if (num_tokens < 0) return fail(PA_ERR_INVALID_ARG, "num_tokens must be >= 0%s");
  if (num_tokens == 0) return ok();
  if (!k || !v || !k_cache || !v_cache || !slot_mapping)
    return fail(PA_ERR_INVALID_ARG, "k, v, k_cache, v_cache and slot_mapping must be non-NULL%s");
  if (!aligned16(k) || !aligned16(v) || !aligned16(k_cache) || !aligned16(v_cache))
    return fail(PA_ERR_INVALID_ARG, "k, v, k_cache and v_cache must be 16-byte aligned%s");
  if (!aligned16(slot_mapping) && (reinterpret_cast<uintptr_t>(slot_mapping) & 7u))
    return fail(PA_ERR_INVALID_ARG, "slot_mapping must be 8-byte aligned%s");
  const cudaError_t e = pa::launch_cache_write(*desc, k, v, k_cache, v_cache, slot_mapping,
                                               num_tokens, reinterpret_cast<cudaStream_t>(stream));
  return e == cudaSuccess ? ok() : cuda_fail(e);
}

size_t pa_decode_workspace_size(const pa_kv_desc *desc, int32_t num_seqs, int32_t max_context_len) {
  (void)max_context_len;
  if (check_desc(desc) != PA_OK || num_seqs < 0) return 0;
  pa::DecodePlan plan;
  const char *why = "";
  if (pa::plan_decode(*desc, num_seqs, &plan, &why) != PA_OK) {
    fail(PA_ERR_UNSUPPORTED, "%s", why);
    return 0;
  }
  return plan.workspace_bytes;
}

pa_status pa_decode(const pa_kv_desc *desc, float *out, float *lse, const void *q,
                    const void *k_cache, const void *v_cache, const int32_t *block_tables,
                    int32_t max_blocks_per_seq, const int32_t *context_lens, int32_t num_seqs,
                    int32_t max_context_len, float scale, void *workspace, size_t workspace_bytes,
                    pa_stream_t stream) {
  pa::DecodePlan plan;
  pa_status st = pa::validate_decode(desc, out, lse, q, k_cache, v_cache, block_tables, max_blocks_per_seq,
                                     context_lens, num_seqs, max_context_len, scale, &plan);
  if (st != PA_OK) return st;
  if (num_seqs == 0) return ok();
  if (!workspace || !aligned16(workspace))
    return fail(PA_ERR_WORKSPACE, "workspace must be non-NULL and 16-byte aligned%s");
  if (workspace_bytes < plan.workspace_bytes)
    return fail(PA_ERR_WORKSPACE, "workspace is smaller than pa_decode_workspace_size()%s");
  const cudaError_t e = pa::launch_decode(*desc, plan, out, lse, q, k_cache, v_cache, block_tables,
                                          max_blocks_per_seq, context_lens, num_seqs, scale,
                                          workspace, reinterpret_cast<cudaStream_t>(stream));
  return e == cudaSuccess ? ok() : cuda_fail(e);
}

pa_status pa_prefill_chunk(const pa_kv_desc *desc, float *out, float *lse, const void *q,
                           const int32_t *query_start_loc, const void *k_cache,
                           const void *v_cache, const int32_t *block_tables,
                           int32_t max_blocks_per_seq, const int32_t *context_lens,
                           int32_t num_seqs, int32_t max_q_len, int32_t max_context_len,
                           float scale, pa_stream_t stream) {
  const pa_status st = pa::validate_prefill(desc, out, lse, q, query_start_loc, k_cache, v_cache, block_tables,
                                            max_blocks_per_seq, context_lens, num_seqs, max_q_len, max_context_len,
                                            scale);
  if (st != PA_OK) return st;
  if (num_seqs == 0 || max_q_len == 0) return ok();
  const cudaError_t e = pa::launch_prefill(*desc, out, lse, q, query_start_loc, k_cache, v_cache,
                                           block_tables, max_blocks_per_seq, context_lens, num_seqs,
                                           max_q_len, scale, reinterpret_cast<cudaStream_t>(stream));
  return e == cudaSuccess ? ok() : cuda_fail(e);
}

int32_t pa_prefill_balanced_chosen(const pa_kv_desc *desc, int32_t num_seqs, int32_t max_q_len,
                                   int32_t max_context_len, int32_t max_blocks_per_seq) {
  if (check_desc(desc) != PA_OK) return -1;
  const char *why = "";
  if (num_seqs < 0 || max_q_len < 0 || max_context_len < 0 || max_blocks_per_seq <= 0 ||
      pa::check_prefill(*desc, &why) != PA_OK)
    return -1;
  if (num_seqs == 0 || max_q_len == 0) return 0;
  return pa::prefill_balanced_chosen(*desc, num_seqs, max_q_len, max_context_len, max_blocks_per_seq) ? 1 : 0;
}

pa_status pa_decode_append(const pa_kv_desc *desc, float *out, float *lse, const void *q, const void *k_new,
                           const void *v_new, void *k_cache, void *v_cache, const int32_t *block_tables,
                           int32_t max_blocks_per_seq, const int32_t *context_lens, int32_t num_seqs,
                           int32_t max_context_len, float scale, void *workspace, size_t workspace_bytes,
                           pa_stream_t stream) {
  static const char *kNotTaken =
      "pa_decode_append runs on the tensor-core decode kernel (with decode_impl PA_DECODE_SIMT make the "
      "pa_cache_write and pa_decode calls instead)%s";
  // the checks that need no device come first
  pa_status st = check_desc(desc);
  if (st != PA_OK) return st;
  if (num_seqs > 0 && (!k_new || !v_new || !aligned16(k_new) || !aligned16(v_new)))
    return fail(PA_ERR_INVALID_ARG, "k_new and v_new must be non-NULL and 16-byte aligned%s");
  pa::DecodePlan plan;
  st = pa::validate_decode(desc, out, lse, q, k_cache, v_cache, block_tables, max_blocks_per_seq, context_lens,
                           num_seqs, max_context_len, scale, &plan);
  if (st != PA_OK) return st;
  if (num_seqs == 0) return ok();
  if (plan.impl != PA_DECODE_MMA) return fail(PA_ERR_UNSUPPORTED, kNotTaken);
  if (!workspace || !aligned16(workspace))
    return fail(PA_ERR_WORKSPACE, "workspace must be non-NULL and 16-byte aligned%s");
  if (workspace_bytes < plan.workspace_bytes)
    return fail(PA_ERR_WORKSPACE, "workspace is smaller than pa_decode_workspace_size()%s");
  const cudaError_t e = pa::launch_decode(*desc, plan, out, lse, q, k_cache, v_cache, block_tables,
                                          max_blocks_per_seq, context_lens, num_seqs, scale, workspace,
                                          reinterpret_cast<cudaStream_t>(stream), k_new, v_new);
  return e == cudaSuccess ? ok() : cuda_fail(e);
}

size_t pa_prefill_workspace_size(const pa_kv_desc *desc, int32_t num_seqs, int32_t max_q_len) {
  if (check_desc(desc) != PA_OK || num_seqs < 0 || max_q_len < 0) return 0;
  const char *why = "";
  if (pa::check_prefill(*desc, &why) != PA_OK) {
    fail(PA_ERR_UNSUPPORTED, "%s", why);
    return 0;
  }
  return pa::prefill_sk_workspace_bytes(*desc, num_seqs, max_q_len);
}

pa_status pa_prefill_chunk_balanced(const pa_kv_desc *desc, float *out, float *lse, const void *q,
                                    const int32_t *query_start_loc, const void *k_cache, const void *v_cache,
                                    const int32_t *block_tables, int32_t max_blocks_per_seq,
                                    const int32_t *context_lens, int32_t num_seqs, int32_t max_q_len,
                                    int32_t max_context_len, float scale, void *workspace, size_t workspace_bytes,
                                    pa_stream_t stream) {
  const pa_status st = pa::validate_prefill(desc, out, lse, q, query_start_loc, k_cache, v_cache, block_tables,
                                            max_blocks_per_seq, context_lens, num_seqs, max_q_len, max_context_len,
                                            scale);
  if (st != PA_OK) return st;
  if (num_seqs == 0 || max_q_len == 0) return ok();
  if (!workspace || !aligned16(workspace))
    return fail(PA_ERR_WORKSPACE, "workspace must be non-NULL and 16-byte aligned%s");
  if (workspace_bytes < pa::prefill_sk_workspace_bytes(*desc, num_seqs, max_q_len))
    return fail(PA_ERR_WORKSPACE, "workspace is smaller than pa_prefill_workspace_size()%s");
  const cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  const bool balanced = pa::prefill_balanced_chosen(*desc, num_seqs, max_q_len, max_context_len, max_blocks_per_seq);
  const cudaError_t e =
      balanced
          ? pa::launch_prefill_tc_sk(*desc, out, lse, q, query_start_loc, k_cache, v_cache, block_tables,
                                     max_blocks_per_seq, context_lens, num_seqs, max_q_len, scale, workspace, s)
          : pa::launch_prefill(*desc, out, lse, q, query_start_loc, k_cache, v_cache, block_tables,
                               max_blocks_per_seq, context_lens, num_seqs, max_q_len, scale, s);
  return e == cudaSuccess ? ok() : cuda_fail(e);
}

size_t pa_mixed_workspace_size(const pa_kv_desc *desc, int32_t num_dec_seqs, int32_t dec_max_context_len) {
  (void)dec_max_context_len;
  if (check_desc(desc) != PA_OK || num_dec_seqs < 0) return 0;
  pa::DecodePlan plan;
  const char *why = "";
  if (pa::plan_decode(*desc, num_dec_seqs, &plan, &why) != PA_OK) {
    fail(PA_ERR_UNSUPPORTED, "%s", why);
    return 0;
  }
  return pa::mixed_plan(*desc, num_dec_seqs, plan).workspace_bytes;
}

namespace {

// pa_mixed_attention and pa_mixed_attention_append: the same checks, and
// the append's new rows (NULL: none)
pa_status mixed_call(const pa_kv_desc *desc, float *dec_out, float *dec_lse, const void *dec_q,
                     const int32_t *dec_block_tables, int32_t dec_max_blocks_per_seq, const int32_t *dec_context_lens,
                     int32_t num_dec_seqs, int32_t dec_max_context_len, float *pf_out, float *pf_lse, const void *pf_q,
                     const int32_t *query_start_loc, const int32_t *pf_block_tables, int32_t pf_max_blocks_per_seq,
                     const int32_t *pf_context_lens, int32_t num_pf_seqs, int32_t max_q_len,
                     int32_t pf_max_context_len, const void *k_cache, const void *v_cache, float scale,
                     void *workspace, size_t workspace_bytes, pa_stream_t stream, bool append, const void *k_new,
                     const void *v_new, int64_t num_new_rows) {
  // the decode part's checks (and its plan, whose workspace the call uses);
  // with no decode sequence only the descriptor and the plan of an empty batch
  pa::DecodePlan plan;
  pa_status st = pa::validate_decode(desc, dec_out, dec_lse, dec_q, k_cache, v_cache, dec_block_tables,
                                     dec_max_blocks_per_seq, dec_context_lens, num_dec_seqs, dec_max_context_len,
                                     scale, &plan);
  if (st != PA_OK) return st;
  if (num_dec_seqs == 0) {
    const char *why = "";
    st = pa::plan_decode(*desc, 0, &plan, &why);
    if (st != PA_OK) return fail(st, "%s", why);
  }
  st = pa::validate_prefill(desc, pf_out, pf_lse, pf_q, query_start_loc, k_cache, v_cache, pf_block_tables,
                            pf_max_blocks_per_seq, pf_context_lens, num_pf_seqs, max_q_len, pf_max_context_len, scale);
  if (st != PA_OK) return st;
  const char *why = "";
  st = pa::check_mixed(*desc, plan, &why);
  if (st != PA_OK) return fail(st, "%s", why);
  const bool has_pf = num_pf_seqs > 0 && max_q_len > 0;
  if (append) {
    if (num_dec_seqs > 0 || has_pf) {
      if (!k_new || !v_new || !aligned16(k_new) || !aligned16(v_new))
        return fail(PA_ERR_INVALID_ARG, "k_new and v_new must be non-NULL and 16-byte aligned%s");
      if (num_new_rows < num_dec_seqs + (has_pf ? 1 : 0))
        return fail(PA_ERR_INVALID_ARG,
                    "num_new_rows must count the decode rows and the prefill chunks' rows of k_new%s");
    }
    if (!has_pf) num_new_rows = num_dec_seqs;
  }
  plan = pa::mixed_plan(*desc, num_dec_seqs, plan);
  if (!workspace || !aligned16(workspace))
    return fail(PA_ERR_WORKSPACE, "workspace must be non-NULL and 16-byte aligned%s");
  if (workspace_bytes < plan.workspace_bytes)
    return fail(PA_ERR_WORKSPACE, "workspace is smaller than pa_mixed_workspace_size()%s");
  const cudaError_t e = pa::launch_mixed(
      *desc, plan, dec_out, dec_lse, dec_q, dec_block_tables, dec_max_blocks_per_seq, dec_context_lens, num_dec_seqs,
      pf_out, pf_lse, pf_q, query_start_loc, pf_block_tables, pf_max_blocks_per_seq, pf_context_lens, num_pf_seqs,
      max_q_len, k_cache, v_cache, scale, workspace, reinterpret_cast<cudaStream_t>(stream),
      append ? k_new : nullptr, append ? v_new : nullptr, append ? num_new_rows : 0);
  return e == cudaSuccess ? ok() : cuda_fail(e);
}

}  // namespace

pa_status pa_mixed_attention(const pa_kv_desc *desc, float *dec_out, float *dec_lse, const void *dec_q,
                             const int32_t *dec_block_tables, int32_t dec_max_blocks_per_seq,
                             const int32_t *dec_context_lens, int32_t num_dec_seqs, int32_t dec_max_context_len,
                             float *pf_out, float *pf_lse, const void *pf_q, const int32_t *query_start_loc,
                             const int32_t *pf_block_tables, int32_t pf_max_blocks_per_seq,
                             const int32_t *pf_context_lens, int32_t num_pf_seqs, int32_t max_q_len,
                             int32_t pf_max_context_len, const void *k_cache, const void *v_cache, float scale,
                             void *workspace, size_t workspace_bytes, pa_stream_t stream) {
  return mixed_call(desc, dec_out, dec_lse, dec_q, dec_block_tables, dec_max_blocks_per_seq, dec_context_lens,
                    num_dec_seqs, dec_max_context_len, pf_out, pf_lse, pf_q, query_start_loc, pf_block_tables,
                    pf_max_blocks_per_seq, pf_context_lens, num_pf_seqs, max_q_len, pf_max_context_len, k_cache,
                    v_cache, scale, workspace, workspace_bytes, stream, false, nullptr, nullptr, 0);
}

pa_status pa_mixed_attention_append(const pa_kv_desc *desc, float *dec_out, float *dec_lse, const void *dec_q,
                                    const int32_t *dec_block_tables, int32_t dec_max_blocks_per_seq,
                                    const int32_t *dec_context_lens, int32_t num_dec_seqs,
                                    int32_t dec_max_context_len, float *pf_out, float *pf_lse, const void *pf_q,
                                    const int32_t *query_start_loc, const int32_t *pf_block_tables,
                                    int32_t pf_max_blocks_per_seq, const int32_t *pf_context_lens,
                                    int32_t num_pf_seqs, int32_t max_q_len, int32_t pf_max_context_len,
                                    const void *k_new, const void *v_new, int64_t num_new_rows, void *k_cache,
                                    void *v_cache, float scale, void *workspace, size_t workspace_bytes,
                                    pa_stream_t stream) {
  return mixed_call(desc, dec_out, dec_lse, dec_q, dec_block_tables, dec_max_blocks_per_seq, dec_context_lens,
                    num_dec_seqs, dec_max_context_len, pf_out, pf_lse, pf_q, query_start_loc, pf_block_tables,
                    pf_max_blocks_per_seq, pf_context_lens, num_pf_seqs, max_q_len, pf_max_context_len, k_cache,
                    v_cache, scale, workspace, workspace_bytes, stream, true, k_new, v_new, num_new_rows);
}

pa_status pa_prefix_attention(const pa_kv_desc *desc, float *out, float *lse, const void *q,
                              const int32_t *query_start_loc, const void *k_cache, const void *v_cache,
                              const int32_t *prefix_tables, int32_t max_blocks_per_prefix,
                              const int32_t *prefix_lens, int32_t num_groups, int32_t max_q_len,
                              int32_t max_prefix_len, int32_t num_splits, int32_t out_slots, float scale,
                              pa_stream_t stream) {
  pa_status st = check_desc(desc);
  if (st != PA_OK) return st;
  if (desc->sliding_window != 0 || desc->attention_chunk != 0)
    return fail(PA_ERR_UNSUPPORTED, "shared-prefix attention takes no local attention (sliding_window, "
                                    "attention_chunk must be 0)%s");
  if (num_groups < 0 || max_q_len < 0) return fail(PA_ERR_INVALID_ARG, "num_groups and max_q_len must be >= 0%s");
  if (num_groups == 0 || max_q_len == 0) return ok();
  if (!out || !lse || !q || !query_start_loc || !k_cache || !v_cache || !prefix_tables || !prefix_lens)
    return fail(PA_ERR_INVALID_ARG,
                "out, lse, q, query_start_loc, k_cache, v_cache, prefix_tables and prefix_lens must be non-NULL%s");
  if (!aligned16(out) || !aligned16(q) || !aligned16(k_cache) || !aligned16(v_cache))
    return fail(PA_ERR_INVALID_ARG, "out, q, k_cache and v_cache must be 16-byte aligned%s");
  if ((reinterpret_cast<uintptr_t>(prefix_tables) & 3u) || (reinterpret_cast<uintptr_t>(prefix_lens) & 3u) ||
      (reinterpret_cast<uintptr_t>(query_start_loc) & 3u) || (reinterpret_cast<uintptr_t>(lse) & 3u))
    return fail(PA_ERR_INVALID_ARG,
                "prefix_tables, prefix_lens, query_start_loc and lse must be 4-byte aligned%s");
  if (max_blocks_per_prefix <= 0) return fail(PA_ERR_INVALID_ARG, "max_blocks_per_prefix must be positive%s");
  if (max_prefix_len < 0 || static_cast<int64_t>(max_prefix_len) > static_cast<int64_t>(max_blocks_per_prefix) * 16)
    return fail(PA_ERR_INVALID_ARG, "max_prefix_len must lie in [0, max_blocks_per_prefix * block_size]%s");
  if (!(scale == scale)) return fail(PA_ERR_INVALID_ARG, "scale is NaN%s");
  if (num_splits < 1 || num_splits > 4096) return fail(PA_ERR_INVALID_ARG, "num_splits must lie in [1, 4096]%s");
  if (out_slots == 0) out_slots = num_splits;
  if (out_slots < num_splits) return fail(PA_ERR_INVALID_ARG, "out_slots must be >= num_splits (or 0)%s");
  if (static_cast<int64_t>(num_groups) * num_splits > 65535)
    return fail(PA_ERR_UNSUPPORTED, "num_groups * num_splits must be at most 65535%s");
  const char *why = "";
  st = pa::check_prefill(*desc, &why);
  if (st != PA_OK) return fail(st, "%s", why);
  // keys per split: a whole number of 128-key tiles
  int split_len = (max_prefix_len + num_splits - 1) / num_splits;
  split_len = split_len < 128 ? 128 : (split_len + 127) / 128 * 128;
  const cudaError_t e = pa::launch_prefill(*desc, out, lse, q, query_start_loc, k_cache, v_cache, prefix_tables,
                                           max_blocks_per_prefix, prefix_lens, num_groups, max_q_len, scale,
                                           reinterpret_cast<cudaStream_t>(stream), /*prefix_mode=*/true,
                                           num_splits, split_len, out_slots);
  return e == cudaSuccess ? ok() : cuda_fail(e);
}

pa_status pa_copy_blocks(const pa_kv_desc *desc, void *k_cache, void *v_cache, const int32_t *src_blocks,
                         const int32_t *dst_blocks, int32_t num_pairs, pa_stream_t stream) {
  pa_status st = check_desc(desc);
  if (st != PA_OK) return st;
  if (num_pairs < 0) return fail(PA_ERR_INVALID_ARG, "num_pairs must be >= 0%s");
  if (num_pairs == 0) return ok();
  if (!k_cache || !v_cache || !src_blocks || !dst_blocks)
    return fail(PA_ERR_INVALID_ARG, "k_cache, v_cache, src_blocks and dst_blocks must be non-NULL%s");
  if (!aligned16(k_cache) || !aligned16(v_cache))
    return fail(PA_ERR_INVALID_ARG, "k_cache and v_cache must be 16-byte aligned%s");
  if ((reinterpret_cast<uintptr_t>(src_blocks) & 3u) || (reinterpret_cast<uintptr_t>(dst_blocks) & 3u))
    return fail(PA_ERR_INVALID_ARG, "src_blocks and dst_blocks must be 4-byte aligned%s");
  const cudaError_t e = pa::launch_copy_blocks(*desc, k_cache, v_cache, src_blocks, dst_blocks, num_pairs,
                                               reinterpret_cast<cudaStream_t>(stream));
  return e == cudaSuccess ? ok() : cuda_fail(e);
}

pa_status pa_bind_blocks(const pa_kv_desc *desc, int32_t *block_tables, int32_t max_blocks_per_seq,
                         int32_t num_table_rows, const int32_t *seq_rows, const int32_t *hit_start,
                         const int32_t *hit_blocks, int32_t num_seqs, int32_t *refcounts, pa_stream_t stream) {
  pa_status st = check_desc(desc);
  if (st != PA_OK) return st;
  if (num_seqs < 0 || num_table_rows < 0) return fail(PA_ERR_INVALID_ARG, "num_seqs and num_table_rows must be >= 0%s");
  if (num_seqs == 0) return ok();
  if (num_seqs > 0x7fffffff / 2) return fail(PA_ERR_UNSUPPORTED, "too many sequences%s");
  if (max_blocks_per_seq <= 0) return fail(PA_ERR_INVALID_ARG, "max_blocks_per_seq must be positive%s");
  if (!block_tables || !seq_rows || !hit_start || !hit_blocks || !refcounts)
    return fail(PA_ERR_INVALID_ARG, "block_tables, seq_rows, hit_start, hit_blocks and refcounts must be non-NULL%s");
  if ((reinterpret_cast<uintptr_t>(block_tables) | reinterpret_cast<uintptr_t>(seq_rows) |
       reinterpret_cast<uintptr_t>(hit_start) | reinterpret_cast<uintptr_t>(hit_blocks) |
       reinterpret_cast<uintptr_t>(refcounts)) & 3u)
    return fail(PA_ERR_INVALID_ARG, "the page-table arrays must be 4-byte aligned%s");
  const cudaError_t e = pa::launch_bind_blocks(*desc, block_tables, max_blocks_per_seq, num_table_rows, seq_rows,
                                               hit_start, hit_blocks, num_seqs, refcounts,
                                               reinterpret_cast<cudaStream_t>(stream));
  return e == cudaSuccess ? ok() : cuda_fail(e);
}

pa_status pa_release_blocks(const pa_kv_desc *desc, int32_t *block_tables, int32_t max_blocks_per_seq,
                            int32_t num_table_rows, const int32_t *seq_rows, const int32_t *block_counts,
                            int32_t num_seqs, int32_t *refcounts, int32_t *free_list, int32_t *free_count,
                            pa_stream_t stream) {
  pa_status st = check_desc(desc);
  if (st != PA_OK) return st;
  if (num_seqs < 0 || num_table_rows < 0) return fail(PA_ERR_INVALID_ARG, "num_seqs and num_table_rows must be >= 0%s");
  if (num_seqs == 0) return ok();
  if (num_seqs > 0x7fffffff / 2) return fail(PA_ERR_UNSUPPORTED, "too many sequences%s");
  if (max_blocks_per_seq <= 0) return fail(PA_ERR_INVALID_ARG, "max_blocks_per_seq must be positive%s");
  if (!block_tables || !seq_rows || !block_counts || !refcounts || !free_list || !free_count)
    return fail(PA_ERR_INVALID_ARG,
                "block_tables, seq_rows, block_counts, refcounts, free_list and free_count must be non-NULL%s");
  if ((reinterpret_cast<uintptr_t>(block_tables) | reinterpret_cast<uintptr_t>(seq_rows) |
       reinterpret_cast<uintptr_t>(block_counts) | reinterpret_cast<uintptr_t>(refcounts) |
       reinterpret_cast<uintptr_t>(free_list) | reinterpret_cast<uintptr_t>(free_count)) & 3u)
    return fail(PA_ERR_INVALID_ARG, "the page-table arrays must be 4-byte aligned%s");
  const cudaError_t e = pa::launch_release_blocks(*desc, block_tables, max_blocks_per_seq, num_table_rows, seq_rows,
                                                  block_counts, num_seqs, refcounts, free_list, free_count,
                                                  reinterpret_cast<cudaStream_t>(stream));
  return e == cudaSuccess ? ok() : cuda_fail(e);
}

pa_status pa_merge_partials(float *out, float *lse_out, const float *part_o,
                            const float *part_lse, const int32_t *num_parts, int32_t num_seqs,
                            int32_t num_heads, int32_t max_parts, int32_t head_dim,
                            pa_stream_t stream) {
  if (num_seqs < 0 || num_heads <= 0 || max_parts < 0)
    return fail(PA_ERR_INVALID_ARG, "num_seqs >= 0, num_heads > 0 and max_parts >= 0 required%s");
  if (head_dim <= 0 || head_dim % 4 != 0 || head_dim > 512)
    return fail(PA_ERR_UNSUPPORTED, "head_dim must be a positive multiple of 4, at most 512%s");
  if (num_seqs == 0) return ok();
  if (!out || (max_parts > 0 && (!part_o || !part_lse)))
    return fail(PA_ERR_INVALID_ARG, "out, part_o and part_lse must be non-NULL%s");
  if (!aligned16(out) || !aligned16(part_o))
    return fail(PA_ERR_INVALID_ARG, "out and part_o must be 16-byte aligned%s");
  if ((reinterpret_cast<uintptr_t>(part_lse) & 3u) || (reinterpret_cast<uintptr_t>(lse_out) & 3u) ||
      (reinterpret_cast<uintptr_t>(num_parts) & 3u))
    return fail(PA_ERR_INVALID_ARG, "part_lse, lse_out and num_parts must be 4-byte aligned%s");
  if (static_cast<int64_t>(num_seqs) * num_heads > 0x7fffffff)
    return fail(PA_ERR_UNSUPPORTED, "num_seqs * num_heads exceeds the grid limit%s");
  const cudaError_t e = pa::launch_merge(out, lse_out, part_o, part_lse, num_parts, num_seqs,
                                         num_heads, max_parts, head_dim,
                                         reinterpret_cast<cudaStream_t>(stream));
  return e == cudaSuccess ? ok() : cuda_fail(e);
}

pa_status pa_test_prefill_schedule(int32_t schedule) {
  if (schedule < 0 || schedule > 2) return fail(PA_ERR_INVALID_ARG, "schedule must be 0, 1 or 2%s");
  g_test_schedule.store(schedule, std::memory_order_relaxed);
  return ok();
}

pa_status pa_test_stall_pipelines(int32_t enable, int64_t wait_limit_ns) {
  if (enable && wait_limit_ns <= 0) return fail(PA_ERR_INVALID_ARG, "wait_limit_ns must be positive%s");
  g_test_wait_ns.store(enable ? static_cast<unsigned long long>(wait_limit_ns) : 0ull, std::memory_order_relaxed);
  g_test_stall.store(enable ? 1 : 0, std::memory_order_relaxed);
  return ok();
}

}  // extern "C"
