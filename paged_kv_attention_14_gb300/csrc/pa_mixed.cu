// pa_mixed.cu -- decode and chunked-prefill attention of one continuous-batch
// step in a single persistent launch (pa_mixed_attention).
//
// The vllm.cpp engine runs decode sequences and prefill chunks in one
// continuously batched step ("C++20 Continuous Batching Loop" in the
// "vllm.cpp ARCHITECTURE OVERVIEW" figure of "Building and Deploying
// vllm.cpp ..."; the unified token-budget scheduler with chunked prefill of
// the vllm.cpp repository's Engine core bullet).  After the step's cache
// write, its decode attention (memory-bound) and prefill attention
// (tensor-bound) read the same cache and write disjoint outputs.
//
// How (GB300 design): one CTA per SM, each taking work items from a flat
// list -- the prefill tiles of the tcgen05 kernel (pa_prefill_tc.cuh),
// longest key ranges first, then the partitions of the decode's stream-K
// split (pa_decode_kernels.cuh) -- through an atomic counter in the decode
// workspace.  Prefill tiles thus keep priority, and the decode fills the SMs
// that the prefill's last wave leaves idle, at the full per-SM bandwidth
// the prefill leaves unused.  Every CTA allocates its tensor memory once;
// both bodies reuse the same shared memory item after item.  The last CTA
// to run out of work resets the counters, so the workspace is ready for the
// next launch.
#include "pa_decode_kernels.cuh"
#include "pa_host_cache.h"
#include "pa_prefill_tc.cuh"

namespace pa {

// Optional item trace (compiled only with -DPA_MIXED_TRACE): per CTA, up to
// 16 items of (item, global-timer start, end).
#ifdef PA_MIXED_TRACE
static __device__ unsigned long long g_mix_trace[256][16][3];
#endif

namespace {

struct MixedArgs {
  pftc::Args pf;        // the prefill part: tiles of a (gx, gy, gz) grid
  dec::DecodeArgs dec;  // the decode part: n_dec partitions
  int pf_gx, pf_gy, pf_gz;
  int n_pf, n_dec;
  int32_t *next_item;   // workspace: the next work item
  int32_t *finished;    // workspace: CTAs that ran out of work
};

// Consumer warps of a decode partition in the single-launch step: a
// partition runs alone on its SM, where four consumer warps stream well
// below the SM's share of the HBM bandwidth; the CTA has 12 warps, and six
// consumers still leave room for three stages (GQ <= 8).
template <int GQ>
constexpr int mixed_decode_warps() {
  return GQ <= 8 ? 6 : dec::kConsumerWarps;
}

template <int D, int KVT, int GQ>
__global__ void __launch_bounds__(pftc::NTHREADS, 1) mixed_kernel(const __grid_constant__ MixedArgs m) {
  constexpr int NCW = mixed_decode_warps<GQ>();
  constexpr int NS = dec::mma_stages<D, KVT, GQ, 1, NCW>();
  // launched as a programmatic dependent of the preceding kernel (the cache
  // write, unless this launch writes the step's rows itself): nothing is
  // read before its writes are visible
  asm volatile("griddepcontrol.wait;" ::: "memory");
  extern __shared__ uint8_t smem_raw[];
  uint8_t *smem = pftc::align1024(smem_raw);
  __shared__ uint32_t s_tmem;
  __shared__ int s_item;
  const int warp = threadIdx.x >> 5;
  if (warp == pftc::kMmaWarp) tmem_alloc(&s_tmem, pftc::Cfg<D, KVT, pftc::kPvF16>::TMEM_COLS);
  tc_fence_before_sync();
  __syncthreads();
  tc_fence_after_sync();
  const uint32_t tmem = s_tmem;
  const int total = m.n_pf + m.n_dec;
#ifdef PA_MIXED_TRACE
  int n_done = 0;
#endif
  for (;;) {
    if (threadIdx.x == 0) s_item = atomicAdd(m.next_item, 1);
    // the previous item's generic writes to shared memory (barriers, data)
    // are ordered before this item's copies into the same bytes
    fence_proxy_async_smem();
    __syncthreads();
    const int item = s_item;
    __syncthreads();  // every thread has read s_item
    if (item >= total) break;
#ifdef PA_MIXED_TRACE
    const unsigned long long t_item = global_timer_ns();
#endif
    if (item < m.n_pf) {
      // x fastest-varying last: the longest key ranges (x = 0) of every
      // (kv head, sequence) first
      const int yz = m.pf_gy * m.pf_gz;
      const int x = item / yz, y = (item % yz) % m.pf_gy, z = (item % yz) / m.pf_gy;
      pftc::prefill_tile<D, KVT, pftc::kPvF16, true>(m.pf, smem, tmem, x, y, z, m.pf_gx);
    } else {
      dec::decode_partition<D, KVT, GQ, 1, NS, NCW>(m.dec, smem_raw, item - m.n_pf, m.n_dec);
    }
    __syncthreads();
#ifdef PA_MIXED_TRACE
    if (threadIdx.x == 0 && blockIdx.x < 256 && n_done < 16) {
      g_mix_trace[blockIdx.x][n_done][0] = item;
      g_mix_trace[blockIdx.x][n_done][1] = t_item;
      g_mix_trace[blockIdx.x][n_done][2] = global_timer_ns();
    }
    ++n_done;
#endif
  }
  if (threadIdx.x == 0) {
    // the last CTA out: every CTA has taken its last item, so the counters
    // can go back to zero for the next launch
    if (atomicAdd(m.finished, 1) == static_cast<int>(gridDim.x) - 1) {
      st_relaxed_gpu(m.next_item, 0);
      st_relaxed_gpu(m.finished, 0);
    }
  }
  tc_fence_before_sync();
  __syncthreads();
  if (warp == pftc::kMmaWarp) {
    tc_fence_after_sync();
    tmem_dealloc(tmem, pftc::Cfg<D, KVT, pftc::kPvF16>::TMEM_COLS);
  }
}

template <int D, int KVT, int GQ>
cudaError_t launch_mixed_t(const MixedArgs &m, cudaStream_t stream) {
  using PC = pftc::Cfg<D, KVT, pftc::kPvF16>;
  constexpr int NCW = mixed_decode_warps<GQ>();
  constexpr int NS = dec::mma_stages<D, KVT, GQ, 1, NCW>();
  static_assert(NS >= 3, "at least three decode stages in flight");
  using DC = dec::MmaCfg<D, KVT, GQ, 1, NS, NCW>;
  constexpr size_t smem = static_cast<size_t>(PC::SMEM_LAUNCH) > DC::SMEM ? static_cast<size_t>(PC::SMEM_LAUNCH)
                                                                             : DC::SMEM;
  static_assert(DC::NTHREADS <= pftc::NTHREADS, "the decode body fits the CTA");
  auto fn = &mixed_kernel<D, KVT, GQ>;
  if (prepare_kernel(reinterpret_cast<const void *>(fn), pftc::NTHREADS, smem) < 1)
    return cudaErrorInvalidConfiguration;
  cudaLaunchAttribute pdl[1];
  pdl[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  pdl[0].val.programmaticStreamSerializationAllowed = 1;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(device_sm_count());
  cfg.blockDim = dim3(pftc::NTHREADS);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = stream;
  cfg.attrs = pdl;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, fn, m);
}

}  // namespace

#ifdef PA_MIXED_TRACE
extern "C" PA_API int pa_debug_mixed_trace_read(unsigned long long *host) {
  return static_cast<int>(cudaMemcpyFromSymbol(host, g_mix_trace, sizeof(unsigned long long) * 256 * 16 * 3));
}
extern "C" PA_API int pa_debug_mixed_trace_clear() {
  static unsigned long long zero[256 * 16 * 3];
  return static_cast<int>(cudaMemcpyToSymbol(g_mix_trace, zero, sizeof zero));
}
#endif

// The decode plan of the single-launch step: kMixedDecodeSplit partitions
// per SM.  A decode partition alone on its SM streams far below its share
// of the HBM bandwidth (about 34 GB/s on GB300, workload 5), so finer
// partitions were tried to spread the decode's tail over more SMs: two per
// SM took 18 us each instead of 28 us, but the per-partition set-up and the
// extra merges grew the total and the step got slower (141 against 133 us
// on workload 5's shapes); one it is.
constexpr int kMixedDecodeSplit = 1;

DecodePlan mixed_plan(const pa_kv_desc &d, int32_t num_dec_seqs, const DecodePlan &plan) {
  DecodePlan p = plan;
  p.num_ctas = plan.num_ctas * kMixedDecodeSplit;
  p.workspace_bytes = dec::ws_layout(num_dec_seqs, p.num_groups, p.num_ctas, p.slot_heads, d.head_dim).total;
  return p;
}

pa_status check_mixed(const pa_kv_desc &d, const DecodePlan &plan, const char **why) {
  if (d.kv_dtype != PA_KV_BF16 && d.kv_dtype != PA_KV_F16) {
    *why = "pa_mixed_attention takes bf16 and fp16 caches";
    return PA_ERR_UNSUPPORTED;
  }
  if (d.head_dim != 128) {
    *why = "pa_mixed_attention takes head_dim 128";
    return PA_ERR_UNSUPPORTED;
  }
  if (plan.impl != PA_DECODE_MMA) {
    *why = "pa_mixed_attention runs the tensor-core decode (decode_impl AUTO or MMA)";
    return PA_ERR_UNSUPPORTED;
  }
  if (d.prefill_impl != PA_PREFILL_AUTO && d.prefill_impl != PA_PREFILL_TCGEN05) {
    *why = "pa_mixed_attention runs the tcgen05 prefill with fp16 P.V (prefill_impl AUTO or TCGEN05)";
    return PA_ERR_UNSUPPORTED;
  }
  return PA_OK;
}

cudaError_t launch_mixed(const pa_kv_desc &d, const DecodePlan &plan, float *dec_out, float *dec_lse,
                         const void *dec_q, const int32_t *dec_block_tables, int32_t dec_max_blocks,
                         const int32_t *dec_context_lens, int32_t num_dec_seqs, float *pf_out, float *pf_lse,
                         const void *pf_q, const int32_t *query_start_loc, const int32_t *pf_block_tables,
                         int32_t pf_max_blocks, const int32_t *pf_context_lens, int32_t num_pf_seqs, int32_t max_q_len,
                         const void *k_cache, const void *v_cache, float scale, void *workspace,
                         cudaStream_t stream, const void *k_new, const void *v_new, int64_t num_new_rows) {
  MixedArgs m;
  memset(&m, 0, sizeof m);
  const int g = d.num_q_heads / d.num_kv_heads;
  if (num_dec_seqs > 0) {
    if (!dec::make_decode_args(d, plan, dec_out, dec_lse, dec_q, k_cache, v_cache, dec_block_tables, dec_max_blocks,
                               dec_context_lens, num_dec_seqs, scale, workspace, &m.dec))
      return cudaErrorInvalidValue;
    m.n_dec = plan.num_ctas;
    if (k_new != nullptr) {
      // the decode sequences' new tokens are rows 0 .. num_dec_seqs - 1:
      // each is written and used by the warp that owns its sequence's last
      // block (see pa_decode_append)
      m.dec.k_new = static_cast<const uint8_t *>(k_new);
      m.dec.v_new = static_cast<const uint8_t *>(v_new);
      m.dec.k_write = static_cast<uint8_t *>(const_cast<void *>(k_cache));
      m.dec.v_write = static_cast<uint8_t *>(const_cast<void *>(v_cache));
      m.dec.k_enc = m.dec.v_enc = 1.f;
    }
  }
  if (num_pf_seqs > 0 && max_q_len > 0) {
    if (!pftc::make_args<128>(&m.pf, d, pf_out, pf_lse, pf_q, query_start_loc, k_cache, v_cache, pf_block_tables,
                              pf_max_blocks, pf_context_lens, scale, false, 1, 0, 1))
      return cudaErrorInvalidValue;
    if (k_new != nullptr) {
      // the chunks' new tokens follow the decode rows, in query order
      const int64_t row_bytes = static_cast<int64_t>(d.num_kv_heads) * d.head_dim * 2;
      const uint8_t *kp = static_cast<const uint8_t *>(k_new) + num_dec_seqs * row_bytes;
      const uint8_t *vp = static_cast<const uint8_t *>(v_new) + num_dec_seqs * row_bytes;
      const int64_t pf_rows = num_new_rows - num_dec_seqs;
      if (!pftc::make_new_rows_map<128>(&m.pf.knmap, kp, pf_rows, d) ||
          !pftc::make_new_rows_map<128>(&m.pf.vnmap, vp, pf_rows, d))
        return cudaErrorInvalidValue;
      m.pf.new_rows = 1;
      m.pf.new_row_count = pf_rows;
      m.pf.k_new = kp;
      m.pf.v_new = vp;
      m.pf.k_write = static_cast<uint8_t *>(const_cast<void *>(k_cache));
      m.pf.v_write = static_cast<uint8_t *>(const_cast<void *>(v_cache));
    }
    m.pf_gx = (max_q_len + m.pf.qt - 1) / m.pf.qt;
    m.pf_gy = d.num_kv_heads;
    m.pf_gz = num_pf_seqs;
    m.n_pf = m.pf_gx * m.pf_gy * m.pf_gz;
  }
  if (m.n_pf + m.n_dec == 0) return cudaSuccess;
  int32_t *head = static_cast<int32_t *>(workspace);
  m.next_item = head + 1;  // after the decode's error word, inside its 256-byte head
  m.finished = head + 2;
  const bool f16 = d.kv_dtype == PA_KV_F16;
  if (g <= 4) return f16 ? launch_mixed_t<128, kKvF16, 4>(m, stream) : launch_mixed_t<128, kKvBf16, 4>(m, stream);
  if (g <= 8) return f16 ? launch_mixed_t<128, kKvF16, 8>(m, stream) : launch_mixed_t<128, kKvBf16, 8>(m, stream);
  return f16 ? launch_mixed_t<128, kKvF16, 16>(m, stream) : launch_mixed_t<128, kKvBf16, 16>(m, stream);
}

}  // namespace pa
