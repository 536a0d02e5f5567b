// pa_prefill_tc.cu -- launch of the tcgen05 chunked-prefill kernel
// (pa_prefill_tc.cuh) for pa_prefill_chunk and pa_prefix_attention: one CTA
// per (query tile, kv head, sequence or sequence x key split).
#include "pa_prefill_tc.cuh"

namespace pa {
namespace pftc {

template <int D, int KVT, int PVM>
cudaError_t launch(const pa_kv_desc &d, float *out, float *lse, const void *q, const int32_t *query_start_loc,
                   const void *k_cache, const void *v_cache, const int32_t *block_tables, int32_t max_blocks_per_seq,
                   const int32_t *context_lens, int32_t num_seqs, int32_t max_q_len, float scale,
                   cudaStream_t stream, bool prefix_mode, int num_splits, int split_len, int out_slots) {
  Args a;
  if (!make_args<D>(&a, d, out, lse, q, query_start_loc, k_cache, v_cache, block_tables, max_blocks_per_seq,
                    context_lens, scale, prefix_mode, num_splits, split_len, out_slots))
    return cudaErrorInvalidValue;
  const int qtiles = (max_q_len + a.qt - 1) / a.qt;
  if (qtiles == 0 || num_seqs == 0) return cudaSuccess;
  auto fn = &prefill_tc_kernel<D, KVT, PVM>;
  if (prepare_kernel(reinterpret_cast<const void *>(fn), NTHREADS, Cfg<D, KVT, PVM>::SMEM_LAUNCH) < 1)
    return cudaErrorInvalidConfiguration;
  cudaLaunchAttribute pdl[1];
  pdl[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  pdl[0].val.programmaticStreamSerializationAllowed = 1;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(qtiles, d.num_kv_heads, num_seqs * a.num_splits);
  cfg.blockDim = dim3(NTHREADS);
  cfg.dynamicSmemBytes = Cfg<D, KVT, PVM>::SMEM_LAUNCH;
  cfg.stream = stream;
  cfg.attrs = pdl;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, fn, a);
}

}  // namespace pftc

#ifdef PA_PREFILL_TIMELINE
extern "C" PA_API int pa_debug_prefill_timeline_read(long long *host) {
  return static_cast<int>(cudaMemcpyFromSymbol(host, pftc::g_pf_tl, sizeof(long long) * 24 * 64));
}
#endif
#ifdef PA_PREFILL_TRACE
extern "C" PA_API int pa_debug_prefill_trace_read(unsigned long long *host, int rows) {
  if (rows > 4096) rows = 4096;
  return static_cast<int>(cudaMemcpyFromSymbol(host, pftc::g_pf_trace, sizeof(unsigned long long) * 16 * rows));
}
#endif

cudaError_t launch_prefill_tc(const pa_kv_desc &d, float *out, float *lse, const void *q,
                              const int32_t *query_start_loc, const void *k_cache, const void *v_cache,
                              const int32_t *block_tables, int32_t max_blocks_per_seq, const int32_t *context_lens,
                              int32_t num_seqs, int32_t max_q_len, float scale, cudaStream_t stream,
                              bool prefix_mode, int num_splits, int split_len, int out_slots, bool pair_p) {
  const bool f16 = d.kv_dtype == PA_KV_F16;
  const bool kv8 = d.kv_dtype == PA_KV_FP8_E4M3 || d.kv_dtype == PA_KV_FP8_E5M2;
  // one instantiation per (head_dim, cache type, P mode)
  auto pick = [&](auto launcher) {
    return launcher(d, out, lse, q, query_start_loc, k_cache, v_cache, block_tables, max_blocks_per_seq,
                    context_lens, num_seqs, max_q_len, scale, stream, prefix_mode, num_splits, split_len, out_slots);
  };
  using namespace pftc;
  if (kv8)  // head_dim 128 and fp16 P (check_prefill)
    return d.kv_dtype == PA_KV_FP8_E5M2 ? pick(launch<128, kKvE5M2, kPvF16>) : pick(launch<128, kKvFp8, kPvF16>);
  if (d.head_dim == 128) {
    if (f16) return pair_p ? pick(launch<128, kKvF16, kPvPair>) : pick(launch<128, kKvF16, kPvF16>);
    return pair_p ? pick(launch<128, kKvBf16, kPvPair>) : pick(launch<128, kKvBf16, kPvF16>);
  }
  if (f16) return pair_p ? pick(launch<64, kKvF16, kPvPair>) : pick(launch<64, kKvF16, kPvF16>);
  return pair_p ? pick(launch<64, kKvBf16, kPvPair>) : pick(launch<64, kKvBf16, kPvF16>);
}

}  // namespace pa
