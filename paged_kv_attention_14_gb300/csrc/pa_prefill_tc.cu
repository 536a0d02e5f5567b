// pa_prefill_tc.cu -- launches of the tcgen05 chunked-prefill kernels
// (pa_prefill_tc.cuh): for pa_prefill_chunk and pa_prefix_attention one CTA
// per (kv head, sequence or sequence x key split, query tile); for
// pa_prefill_chunk_balanced one CTA per SM sharing all items' KV iterations.
#include "pa_prefill_sk.cuh"

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
  if (qtiles > 65535 || static_cast<long long>(num_seqs) * a.num_splits > 65535) return cudaErrorInvalidConfiguration;
  auto fn = &prefill_tc_kernel<D, KVT, PVM>;
  if (prepare_kernel(reinterpret_cast<const void *>(fn), NTHREADS, Cfg<D, KVT, PVM>::SMEM_LAUNCH) < 1)
    return cudaErrorInvalidConfiguration;
  cudaLaunchAttribute pdl[1];
  pdl[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  pdl[0].val.programmaticStreamSerializationAllowed = 1;
  cudaLaunchConfig_t cfg = {};
  // longest key ranges first across the grid: the query tile is the slowest index
  cfg.gridDim = dim3(d.num_kv_heads, num_seqs * a.num_splits, qtiles);
  cfg.blockDim = dim3(NTHREADS);
  cfg.dynamicSmemBytes = Cfg<D, KVT, PVM>::SMEM_LAUNCH;
  cfg.stream = stream;
  cfg.attrs = pdl;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, fn, a);
}

// The balanced launch's workspace: the error word, then the items' piece
// counters (one int32 per (pair, kv head)), then two slots per CTA: the
// pieces' log-sum-exp and their normalised outputs.  Every part starts on a
// 256-byte boundary.
struct SkLayout {
  size_t counters, lse, o, total;
};

inline size_t round256(size_t x) { return (x + 255) & ~size_t(255); }

inline SkLayout sk_layout(int head_dim, long long pairs, int num_kv_heads, int G) {
  SkLayout l;
  l.counters = 256;
  l.lse = l.counters + round256(static_cast<size_t>(pairs) * num_kv_heads * sizeof(int32_t));
  l.o = l.lse + round256(static_cast<size_t>(2) * G * MROWS * sizeof(float));
  l.total = l.o + static_cast<size_t>(2) * G * MROWS * head_dim * sizeof(float);
  return l;
}

template <int D, int KVT, int PVM>
cudaError_t launch_sk(const pa_kv_desc &d, float *out, float *lse, const void *q, const int32_t *query_start_loc,
                      const void *k_cache, const void *v_cache, const int32_t *block_tables,
                      int32_t max_blocks_per_seq, const int32_t *context_lens, int32_t num_seqs, int32_t max_q_len,
                      float scale, void *workspace, cudaStream_t stream) {
  Args a;
  if (!make_args<D>(&a, d, out, lse, q, query_start_loc, k_cache, v_cache, block_tables, max_blocks_per_seq,
                    context_lens, scale, false, 1, 0, 1))
    return cudaErrorInvalidValue;
  const int gx = (max_q_len + a.qt - 1) / a.qt;
  if (gx == 0 || num_seqs == 0) return cudaSuccess;
  const int G = device_sm_count();
  const SkLayout l = sk_layout(D, static_cast<long long>(num_seqs) * gx, d.num_kv_heads, G);
  uint8_t *w = static_cast<uint8_t *>(workspace);
  a.num_seqs = num_seqs;
  a.gx = gx;
  a.ws_err = reinterpret_cast<int32_t *>(w);
  a.part_count = reinterpret_cast<int *>(w + l.counters);
  a.part_lse = reinterpret_cast<float *>(w + l.lse);
  a.part_o = reinterpret_cast<float *>(w + l.o);
  auto fn = &prefill_sk_kernel<D, KVT, PVM>;
  if (prepare_kernel(reinterpret_cast<const void *>(fn), NTHREADS, Cfg<D, KVT, PVM>::SMEM_LAUNCH) < 1)
    return cudaErrorInvalidConfiguration;
  cudaLaunchAttribute pdl[1];
  pdl[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  pdl[0].val.programmaticStreamSerializationAllowed = 1;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(G);
  cfg.blockDim = dim3(NTHREADS);
  cfg.dynamicSmemBytes = Cfg<D, KVT, PVM>::SMEM_LAUNCH;
  cfg.stream = stream;
  cfg.attrs = pdl;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, fn, a);
}

}  // namespace pftc

static long long sk_pairs(const pa_kv_desc &d, int32_t num_seqs, int32_t max_q_len) {
  const int qt = pftc::MROWS / (d.num_q_heads / d.num_kv_heads);
  return static_cast<long long>(num_seqs) * ((max_q_len + qt - 1) / qt);
}

bool prefill_sk_applies(const pa_kv_desc &d, int32_t num_seqs, int32_t max_q_len) {
  const int impl = prefill_impl_of(d);
  if (impl != PA_PREFILL_TCGEN05 && impl != PA_PREFILL_TCGEN05_PAIR) return false;
  const long long pairs = sk_pairs(d, num_seqs, max_q_len);
  return pairs > 0 && pairs <= kPrefillSkMaxPairs;
}

bool prefill_sk_units_fit(const pa_kv_desc &d, int32_t num_seqs, int32_t max_q_len, int32_t max_blocks_per_seq) {
  // KV iterations of an item: at most one per 128 keys its table can hold, plus one
  const long long per_item = static_cast<long long>(max_blocks_per_seq) * 16 / pftc::KT + 2;
  return sk_pairs(d, num_seqs, max_q_len) * d.num_kv_heads * per_item < (1LL << 31);
}

bool prefill_sk_pays(const pa_kv_desc &d, int32_t num_seqs, int32_t max_q_len, int32_t max_context_len) {
  // measured on GB300 (bf16, head_dim 128): a KV tile takes ~2 us of a CTA,
  // and each CTA of the balanced kernel spends ~15-25 us more on its pieces'
  // outputs and merges; the grid's longest item bounds its time.  So the
  // balanced kernel pays when the grid fills less than one wave and the
  // idle SMs' share of its longest item is above ~12 tiles.
  const int sms = device_sm_count();
  const long long items = sk_pairs(d, num_seqs, max_q_len) * d.num_kv_heads;
  if (items >= sms) return false;
  const long long tiles = (static_cast<long long>(max_context_len) + pftc::KT - 1) / pftc::KT;
  return tiles * (sms - items) > 12LL * sms;
}

size_t prefill_sk_workspace_bytes(const pa_kv_desc &d, int32_t num_seqs, int32_t max_q_len) {
  // a batch that runs the plain grid needs the error word only
  if (!prefill_sk_applies(d, num_seqs, max_q_len)) return 256;
  return pftc::sk_layout(d.head_dim, sk_pairs(d, num_seqs, max_q_len), d.num_kv_heads, device_sm_count()).total;
}

cudaError_t launch_prefill_tc_sk(const pa_kv_desc &d, float *out, float *lse, const void *q,
                                 const int32_t *query_start_loc, const void *k_cache, const void *v_cache,
                                 const int32_t *block_tables, int32_t max_blocks_per_seq,
                                 const int32_t *context_lens, int32_t num_seqs, int32_t max_q_len, float scale,
                                 void *workspace, cudaStream_t stream) {
  const bool f16 = d.kv_dtype == PA_KV_F16;
  const bool kv8 = d.kv_dtype == PA_KV_FP8_E4M3 || d.kv_dtype == PA_KV_FP8_E5M2;
  const bool pair_p = prefill_impl_of(d) == PA_PREFILL_TCGEN05_PAIR;
  auto pick = [&](auto launcher) {
    return launcher(d, out, lse, q, query_start_loc, k_cache, v_cache, block_tables, max_blocks_per_seq,
                    context_lens, num_seqs, max_q_len, scale, workspace, stream);
  };
  using namespace pftc;
  if (kv8)
    return d.kv_dtype == PA_KV_FP8_E5M2 ? pick(launch_sk<128, kKvE5M2, kPvF16>) : pick(launch_sk<128, kKvFp8, kPvF16>);
  if (d.head_dim == 128) {
    if (f16) return pair_p ? pick(launch_sk<128, kKvF16, kPvPair>) : pick(launch_sk<128, kKvF16, kPvF16>);
    return pair_p ? pick(launch_sk<128, kKvBf16, kPvPair>) : pick(launch_sk<128, kKvBf16, kPvF16>);
  }
  if (f16) return pair_p ? pick(launch_sk<64, kKvF16, kPvPair>) : pick(launch_sk<64, kKvF16, kPvF16>);
  return pair_p ? pick(launch_sk<64, kKvBf16, kPvPair>) : pick(launch_sk<64, kKvBf16, kPvF16>);
}

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
