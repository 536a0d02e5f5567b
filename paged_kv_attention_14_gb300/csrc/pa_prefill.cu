// pa_prefill.cu -- causal chunked-prefill attention over the paged KV cache.
//
// What it computes: sequence s brings q_len new queries (a "chunked prefill"
// chunk, vllm.cpp implementation notes, Engine core bullet) whose K/V were
// already written into its blocks; query i sits at position
// context_lens[s] - q_len + i and attends keys [0, position] through the
// block table.  Leading blocks may be shared with other sequences after a
// prefix-cache hit ("Zero-Copy Cache Hits" of "1. Technical Mechanics of the
// Radix Cache" in "Building and Deploying vllm.cpp ..."); they are only read.
//
// How (GB300 design): one CTA takes QT consecutive queries of one sequence
// for all g query heads of one kv head, so the M rows of its tile are
// (query, head) pairs and every K/V tile is loaded once for the whole GQA
// group.  64-key K/V tiles are gathered block by block through the block
// table with 16-byte cp.async into XOR-swizzled shared memory (double
// buffered), then QK^T and PV run on the tensor cores as bf16 (fp16 for an
// fp16 cache) m16n8k16 MMAs with fp32 accumulators and online softmax in
// registers; the probabilities enter PV as a hi + lo pair so the result
// keeps near-fp32 accuracy.  Keys past the sequence end are zero-filled, so
// poisoned tails never reach an MMA; the causal mask is applied only on
// tiles that cross the diagonal.  FP8 tiles are staged raw and decoded to
// bf16 in shared memory (exact: every E4M3 / E5M2 value is a bf16 value),
// with k_scale folded into the softmax scale and v_scale into the output
// (per kv head where the cache has per-head scales).  Local attention
// starts the key walk at the tile of the first visible key.  In prefix mode
// (pa_prefix_attention) every query comes after all the keys of its split
// of a shared prefix, and the outputs go to that split's part slot.
#include "pa_device.cuh"
#include "pa_host_cache.h"
#include "pa_internal.h"

namespace pa {

namespace {

constexpr float kLog2e = 1.4426950408889634f;
constexpr float kLn2 = 0.6931471805599453f;

struct PrefillArgs {
  float *out;
  float *lse;
  const uint16_t *q;
  const int32_t *query_start_loc;
  const uint8_t *k_cache;
  const uint8_t *v_cache;
  const int32_t *block_tables;
  const int32_t *context_lens;
  int max_blocks_per_seq;
  int num_kv_heads;
  int num_q_heads;
  int g;
  int qt;  // queries per CTA
  float qscale;
  float vscale;
  float qscale0;  // scale * log2(e): qscale before the k scale
  const float *k_scales;  // per-kv-head scales of an 8-bit cache (NULL: per-tensor)
  const float *v_scales;
  int window;  // local attention (see pa_kv_desc), 0: none
  int chunk;
  int prefix_mode;  // 1: every query after all L keys, no causal mask (shared prefix)
  int num_splits;   // prefix mode: key splits per sequence (grid.z = sequences x splits)
  int split_len;    // prefix mode: keys per split (a multiple of 128)
  int out_slots;    // prefix mode: output slots per (row, head); split i writes slot i
  int32_t *err;     // the caller's error word (pa_kv_desc.error_word), or NULL
  int checked;      // range-check block ids and lengths (pa_kv_desc.check_indices)
  int num_blocks;   // blocks of the cache (checked mode)
};

template <int D, int KVT, int NW>
struct PrefillCfg {
  static constexpr int KT = 64;                 // keys per tile
  static constexpr int NT = NW * 32;
  static constexpr int CH = D / 8;              // 16-byte bf16 chunks per row
  static constexpr int TILE = KT * D * 2;       // bf16 tile bytes
  static constexpr int RAW = KT * D;            // E4M3 tile bytes
  static constexpr size_t SMEM = kv16(KVT) ? size_t(4) * TILE : size_t(2) * TILE + size_t(4) * RAW;
  // element type of the MMAs: fp16 for an fp16 cache; bf16 for bf16 and for
  // the 8-bit caches, whose tiles are decoded to bf16 in shared memory
  static constexpr int MT16 = KVT == kKvF16 ? kKvF16 : kKvBf16;
};

// byte offset of 16-byte chunk `ch` of row `key` in a swizzled bf16 tile
template <int D>
__device__ __forceinline__ int swz(int key, int ch) {
  return key * (D * 2) + ((ch ^ (key & 7)) << 4);
}

template <int D, int KVT, int NW>
__global__ void __launch_bounds__(NW * 32, 1) prefill_kernel(const PrefillArgs a) {
  using C = PrefillCfg<D, KVT, NW>;
  extern __shared__ __align__(128) uint8_t smem[];
  const int split = a.prefix_mode ? static_cast<int>(blockIdx.z) % a.num_splits : 0;
  const int s = a.prefix_mode ? static_cast<int>(blockIdx.z) / a.num_splits : static_cast<int>(blockIdx.z);
  const int kvh = blockIdx.y;
  const int qtile = gridDim.x - 1 - blockIdx.x;  // longest key ranges first
  const int qs = __ldg(a.query_start_loc + s);
  int q_len = __ldg(a.query_start_loc + s + 1) - qs;
  int L = __ldg(a.context_lens + s);
  if (a.checked) {
    // lengths within the table's capacity; a chunk no longer than its context
    // nor than the launch's query tiles; rows start at a row >= 0
    L = checked_len(L, a.max_blocks_per_seq * 16, a.err, nullptr);
    q_len = checked_len(q_len, a.prefix_mode ? static_cast<int>(gridDim.x) * a.qt
                                             : min(L, static_cast<int>(gridDim.x) * a.qt), a.err, nullptr);
    if (qs < 0) {
      if (threadIdx.x == 0) report_error(a.err, nullptr, kErrBadIndex);
      return;
    }
  }
  const int qt0 = qtile * a.qt;
  if (qt0 >= q_len) return;
  const int nq = min(a.qt, q_len - qt0);  // queries of this CTA
  // prefix mode: this CTA's split covers prefix keys [p_lo, p_hi), and every
  // query comes after them all; otherwise query i sits at L - q_len + i
  const int p_lo = a.prefix_mode ? min(L, split * a.split_len) : 0;
  const int p_hi = a.prefix_mode ? min(L, p_lo + a.split_len) : 0;
  const int base_pos = a.prefix_mode ? p_hi - 1 : L - q_len + qt0;  // position of query qt0
  const int kv_end = a.prefix_mode ? p_hi : base_pos + nq;         // keys [kv_lo, kv_end) are needed
  // local attention: the CTA's earliest query sees keys from kv_lo on (the
  // first key never decreases with the position); its latest from lo_max
  const int kv_lo = a.prefix_mode ? p_lo : local_first_key(base_pos, a.window, a.chunk);
  const int lo_max = a.prefix_mode ? p_lo : local_first_key(kv_end - 1, a.window, a.chunk);
  const int kt0 = kv_lo / C::KT;
  const int n_tiles = (kv_end + C::KT - 1) / C::KT;
  const int tid = threadIdx.x;
  const int warp = tid >> 5;
  const int lane = tid & 31;
  const int g = a.g;
  const int32_t *table = a.block_tables + static_cast<int64_t>(s) * a.max_blocks_per_seq;
  // score scale of this CTA's kv head (its own k scale where the cache has per-head scales)
  const float qscale = a.k_scales ? a.qscale0 * __ldg(a.k_scales + kvh) : a.qscale;

  uint8_t *kt_s[2], *vt_s[2];
  uint8_t *kraw[2], *vraw[2];
  if (kv16(KVT)) {
    kt_s[0] = smem;
    vt_s[0] = smem + C::TILE;
    kt_s[1] = smem + 2 * C::TILE;
    vt_s[1] = smem + 3 * C::TILE;
  } else {
    kt_s[0] = kt_s[1] = smem;
    vt_s[0] = vt_s[1] = smem + C::TILE;
    kraw[0] = smem + 2 * C::TILE;
    vraw[0] = kraw[0] + C::RAW;
    kraw[1] = vraw[0] + C::RAW;
    vraw[1] = kraw[1] + C::RAW;
  }

  // gather one 64-key tile (zero-filled outside [kv_lo, kv_end)) into buffer `b`
  auto load_tile = [&](int kt, int b) {
    if (kv16(KVT)) {
      for (int i = tid; i < C::KT * C::CH; i += C::NT) {
        const int key = i / C::CH;
        const int ch = i - key * C::CH;
        const int t = kt * C::KT + key;
        const bool ok = t < kv_end && t >= kv_lo;
        int64_t off = 0;
        if (ok) {
          int phys = __ldg(table + (t >> 4));
          if (a.checked) phys = checked_block(phys, a.num_blocks, a.err, nullptr);
          off = ((static_cast<int64_t>(phys) * a.num_kv_heads + kvh) * 16 + (t & 15)) * (D * 2) + ch * 16;
        }
        cp_async16(kt_s[b] + swz<D>(key, ch), a.k_cache + off, ok);
        cp_async16(vt_s[b] + swz<D>(key, ch), a.v_cache + off, ok);
      }
    } else {
      constexpr int RCH = D / 16;  // 16-byte chunks of an E4M3 row
      for (int i = tid; i < C::KT * RCH; i += C::NT) {
        const int key = i / RCH;
        const int ch = i - key * RCH;
        const int t = kt * C::KT + key;
        const bool ok = t < kv_end && t >= kv_lo;
        int64_t off = 0;
        if (ok) {
          int phys = __ldg(table + (t >> 4));
          if (a.checked) phys = checked_block(phys, a.num_blocks, a.err, nullptr);
          off = ((static_cast<int64_t>(phys) * a.num_kv_heads + kvh) * 16 + (t & 15)) * D + ch * 16;
        }
        cp_async16(kraw[b] + key * D + ch * 16, a.k_cache + off, ok);
        cp_async16(vraw[b] + key * D + ch * 16, a.v_cache + off, ok);
      }
    }
    cp_async_commit();
  };
  // E4M3 raw tile -> swizzled bf16 tile
  auto convert_tile = [&](int b) {
    constexpr int RCH = D / 16;
    for (int i = tid; i < C::KT * RCH; i += C::NT) {
      const int key = i / RCH;
      const int ch = i - key * RCH;
#pragma unroll
      for (int kv = 0; kv < 2; ++kv) {
        const uint4 u = *reinterpret_cast<const uint4 *>((kv ? vraw[b] : kraw[b]) + key * D + ch * 16);
        const uint32_t w[4] = {u.x, u.y, u.z, u.w};
        uint32_t o[8];
#pragma unroll
        for (int c = 0; c < 4; ++c) {
          float f0, f1, f2, f3;
          fp8x2_to_f32<KVT>(static_cast<uint16_t>(w[c] & 0xffffu), f0, f1);
          fp8x2_to_f32<KVT>(static_cast<uint16_t>(w[c] >> 16), f2, f3);
          o[2 * c] = pack_bf16x2(f0, f1);
          o[2 * c + 1] = pack_bf16x2(f2, f3);
        }
        uint8_t *dst = kv ? vt_s[0] : kt_s[0];
        *reinterpret_cast<uint4 *>(dst + swz<D>(key, 2 * ch)) = make_uint4(o[0], o[1], o[2], o[3]);
        *reinterpret_cast<uint4 *>(dst + swz<D>(key, 2 * ch + 1)) = make_uint4(o[4], o[5], o[6], o[7]);
      }
    }
  };

  load_tile(kt0, kt0 & 1);

  // ---- Q fragments of this warp's 16 rows (row = query * g + head)
  const int r_lo = warp * 16 + (lane >> 2);
  const int r_hi = r_lo + 8;
  const int c4 = lane & 3;
  const int rows_used = a.qt * g;
  auto row_query = [&](int r) { return r / g; };
  const bool ok_lo = r_lo < rows_used && row_query(r_lo) < nq;
  const bool ok_hi = r_hi < rows_used && row_query(r_hi) < nq;
  const uint16_t *q_lo = a.q + (static_cast<int64_t>(qs + qt0 + (ok_lo ? row_query(r_lo) : 0)) * a.num_q_heads + kvh * g + (ok_lo ? r_lo % g : 0)) * D;
  const uint16_t *q_hi = a.q + (static_cast<int64_t>(qs + qt0 + (ok_hi ? row_query(r_hi) : 0)) * a.num_q_heads + kvh * g + (ok_hi ? r_hi % g : 0)) * D;
  uint32_t qa[D / 16][4];
#pragma unroll
  for (int ks = 0; ks < D / 16; ++ks) {
    const int d0 = ks * 16 + 2 * c4;
    qa[ks][0] = ok_lo ? __ldg(reinterpret_cast<const uint32_t *>(q_lo + d0)) : 0u;
    qa[ks][1] = ok_hi ? __ldg(reinterpret_cast<const uint32_t *>(q_hi + d0)) : 0u;
    qa[ks][2] = ok_lo ? __ldg(reinterpret_cast<const uint32_t *>(q_lo + d0 + 8)) : 0u;
    qa[ks][3] = ok_hi ? __ldg(reinterpret_cast<const uint32_t *>(q_hi + d0 + 8)) : 0u;
  }
  // causal limit of each row (keys <= pos); invalid rows see no key; first
  // key of each row under local attention
  const int pos_lo = ok_lo ? (a.prefix_mode ? base_pos : base_pos + row_query(r_lo)) : -1;
  const int pos_hi = ok_hi ? (a.prefix_mode ? base_pos : base_pos + row_query(r_hi)) : -1;
  const int first_lo = a.prefix_mode ? p_lo : local_first_key(pos_lo, a.window, a.chunk);
  const int first_hi = a.prefix_mode ? p_lo : local_first_key(pos_hi, a.window, a.chunk);
  // the lowest position of any row of the CTA: tiles entirely below it need no mask
  const int pos_min = base_pos;

  float oacc[D / 8][4];
#pragma unroll
  for (int n = 0; n < D / 8; ++n) oacc[n][0] = oacc[n][1] = oacc[n][2] = oacc[n][3] = 0.f;
  float m_lo = -INFINITY, m_hi = -INFINITY, l_lo = 0.f, l_hi = 0.f;

  for (int kt = kt0; kt < n_tiles; ++kt) {
    const int b = kv16(KVT) ? (kt & 1) : 0;
    if (kt + 1 < n_tiles) {
      load_tile(kt + 1, (kt + 1) & 1);
      cp_async_wait<1>();
    } else {
      cp_async_wait<0>();
    }
    __syncthreads();
    if (!kv16(KVT)) {
      convert_tile(kt & 1);
      __syncthreads();
    }
    const uint32_t ks_base = smem_u32(kt_s[b]);
    const uint32_t vs_base = smem_u32(vt_s[b]);

    // S = Q K^T for 16 rows x 64 keys
    float sacc[8][4];
#pragma unroll
    for (int n = 0; n < 8; ++n) sacc[n][0] = sacc[n][1] = sacc[n][2] = sacc[n][3] = 0.f;
    {
      const int mat = lane >> 3;
      const int rr = lane & 7;
#pragma unroll
      for (int ks = 0; ks < D / 16; ++ks) {
#pragma unroll
        for (int np = 0; np < 4; ++np) {
          const int key = np * 16 + rr + (mat >> 1) * 8;
          const int ch = ks * 2 + (mat & 1);
          uint32_t b0, b1, b2, b3;
          ldmatrix_x4(b0, b1, b2, b3, ks_base + swz<D>(key, ch));
          mma16_16816<C::MT16>(sacc[2 * np], qa[ks][0], qa[ks][1], qa[ks][2], qa[ks][3], b0, b1);
          mma16_16816<C::MT16>(sacc[2 * np + 1], qa[ks][0], qa[ks][1], qa[ks][2], qa[ks][3], b2, b3);
        }
      }
    }
    // scale, mask, row max
    const bool need_mask = kt * C::KT + C::KT - 1 > pos_min || kt * C::KT < lo_max;
    float mx_lo = -INFINITY, mx_hi = -INFINITY;
#pragma unroll
    for (int n = 0; n < 8; ++n) {
#pragma unroll
      for (int e = 0; e < 2; ++e) {
        const int t = kt * C::KT + n * 8 + 2 * c4 + e;
        float vlo = sacc[n][e] * qscale;
        float vhi = sacc[n][2 + e] * qscale;
        if (need_mask) {
          vlo = (t <= pos_lo && t >= first_lo) ? vlo : -INFINITY;
          vhi = (t <= pos_hi && t >= first_hi) ? vhi : -INFINITY;
        }
        sacc[n][e] = vlo;
        sacc[n][2 + e] = vhi;
        mx_lo = fmaxf(mx_lo, vlo);
        mx_hi = fmaxf(mx_hi, vhi);
      }
    }
    mx_lo = fmaxf(mx_lo, __shfl_xor_sync(0xffffffffu, mx_lo, 1));
    mx_lo = fmaxf(mx_lo, __shfl_xor_sync(0xffffffffu, mx_lo, 2));
    mx_hi = fmaxf(mx_hi, __shfl_xor_sync(0xffffffffu, mx_hi, 1));
    mx_hi = fmaxf(mx_hi, __shfl_xor_sync(0xffffffffu, mx_hi, 2));
    const float mn_lo = fmaxf(m_lo, mx_lo);
    const float mn_hi = fmaxf(m_hi, mx_hi);
    const float ref_lo = mn_lo == -INFINITY ? 0.f : mn_lo;
    const float ref_hi = mn_hi == -INFINITY ? 0.f : mn_hi;
    const float corr_lo = exp2f(m_lo - ref_lo);
    const float corr_hi = exp2f(m_hi - ref_hi);
    m_lo = mn_lo;
    m_hi = mn_hi;
    l_lo *= corr_lo;
    l_hi *= corr_hi;
#pragma unroll
    for (int n = 0; n < D / 8; ++n) {
      oacc[n][0] *= corr_lo;
      oacc[n][1] *= corr_lo;
      oacc[n][2] *= corr_hi;
      oacc[n][3] *= corr_hi;
    }
    // P as hi + lo parts of the MMA type: p = hi + lo to about 2^-17 relative
    // (bf16; closer for fp16), so PV keeps close to fp32 accuracy
    uint32_t ph[4][4], pl[4][4];
#pragma unroll
    for (int n = 0; n < 8; ++n) {
      const float p0 = exp2f(sacc[n][0] - ref_lo);
      const float p1 = exp2f(sacc[n][1] - ref_lo);
      const float p2 = exp2f(sacc[n][2] - ref_hi);
      const float p3 = exp2f(sacc[n][3] - ref_hi);
      l_lo += p0 + p1;
      l_hi += p2 + p3;
      const int kk = n >> 1;
      const int i0 = (n & 1) ? 2 : 0;
      const uint32_t h01 = pack16x2<C::MT16>(p0, p1);
      const uint32_t h23 = pack16x2<C::MT16>(p2, p3);
      ph[kk][i0] = h01;
      ph[kk][i0 + 1] = h23;
      pl[kk][i0] = pack16x2<C::MT16>(p0 - lo16<C::MT16>(h01), p1 - hi16<C::MT16>(h01));
      pl[kk][i0 + 1] = pack16x2<C::MT16>(p2 - lo16<C::MT16>(h23), p3 - hi16<C::MT16>(h23));
    }
    // O += P V
    {
      const int mat = lane >> 3;
      const int rr = lane & 7;
#pragma unroll
      for (int kk = 0; kk < 4; ++kk) {
#pragma unroll
        for (int np = 0; np < D / 16; ++np) {
          const int key = kk * 16 + rr + (mat & 1) * 8;
          const int ch = np * 2 + (mat >> 1);
          uint32_t b0, b1, b2, b3;
          ldmatrix_x4_trans(b0, b1, b2, b3, vs_base + swz<D>(key, ch));
          mma16_16816<C::MT16>(oacc[2 * np], ph[kk][0], ph[kk][1], ph[kk][2], ph[kk][3], b0, b1);
          mma16_16816<C::MT16>(oacc[2 * np + 1], ph[kk][0], ph[kk][1], ph[kk][2], ph[kk][3], b2, b3);
          mma16_16816<C::MT16>(oacc[2 * np], pl[kk][0], pl[kk][1], pl[kk][2], pl[kk][3], b0, b1);
          mma16_16816<C::MT16>(oacc[2 * np + 1], pl[kk][0], pl[kk][1], pl[kk][2], pl[kk][3], b2, b3);
        }
      }
    }
    __syncthreads();  // buffer b is refilled by the next iteration's load
  }

  // ---- normalise and store
  l_lo += __shfl_xor_sync(0xffffffffu, l_lo, 1);
  l_lo += __shfl_xor_sync(0xffffffffu, l_lo, 2);
  l_hi += __shfl_xor_sync(0xffffffffu, l_hi, 1);
  l_hi += __shfl_xor_sync(0xffffffffu, l_hi, 2);
  const float vscale = a.v_scales ? __ldg(a.v_scales + kvh) : a.vscale;
  const float inv_lo = l_lo > 0.f ? vscale / l_lo : 0.f;
  const float inv_hi = l_hi > 0.f ? vscale / l_hi : 0.f;
  if (ok_lo) {
    const int64_t row = (static_cast<int64_t>(qs + qt0 + row_query(r_lo)) * a.num_q_heads + kvh * g + r_lo % g) *
                            a.out_slots + split;
    float *o = a.out + row * D;
#pragma unroll
    for (int n = 0; n < D / 8; ++n)
      *reinterpret_cast<float2 *>(o + n * 8 + 2 * c4) = make_float2(oacc[n][0] * inv_lo, oacc[n][1] * inv_lo);
    if (a.lse && c4 == 0) a.lse[row] = (m_lo + log2f(l_lo)) * kLn2;
  }
  if (ok_hi) {
    const int64_t row = (static_cast<int64_t>(qs + qt0 + row_query(r_hi)) * a.num_q_heads + kvh * g + r_hi % g) *
                            a.out_slots + split;
    float *o = a.out + row * D;
#pragma unroll
    for (int n = 0; n < D / 8; ++n)
      *reinterpret_cast<float2 *>(o + n * 8 + 2 * c4) = make_float2(oacc[n][2] * inv_hi, oacc[n][3] * inv_hi);
    if (a.lse && c4 == 0) a.lse[row] = (m_hi + log2f(l_hi)) * kLn2;
  }
}

constexpr int kPrefillWarps = 8;

template <int D, int KVT>
void *prefill_fn() {
  return reinterpret_cast<void *>(&prefill_kernel<D, KVT, kPrefillWarps>);
}

}  // namespace

pa_status check_prefill(const pa_kv_desc &d, const char **why) {
  const int g = d.num_q_heads / d.num_kv_heads;
  if (g > kPrefillWarps * 16) {
    *why = "prefill supports group sizes up to 128";
    return PA_ERR_UNSUPPORTED;
  }
  if (d.prefill_impl < PA_PREFILL_AUTO || d.prefill_impl > PA_PREFILL_TCGEN05_PAIR) {
    *why = "prefill_impl must be PA_PREFILL_AUTO, PA_PREFILL_MMA_SYNC, PA_PREFILL_TCGEN05 or PA_PREFILL_TCGEN05_PAIR";
    return PA_ERR_INVALID_ARG;
  }
  const bool kv8 = d.kv_dtype == PA_KV_FP8_E4M3 || d.kv_dtype == PA_KV_FP8_E5M2;
  if (d.prefill_impl == PA_PREFILL_TCGEN05 && kv8 && d.head_dim != 128) {
    *why = "the tcgen05 prefill kernel takes 8-bit caches with head_dim 128";
    return PA_ERR_UNSUPPORTED;
  }
  if (d.prefill_impl == PA_PREFILL_TCGEN05_PAIR && kv8) {
    *why = "the tcgen05 prefill's pair mode takes bf16 and fp16 caches";
    return PA_ERR_UNSUPPORTED;
  }
  return PA_OK;
}

int prefill_impl_of(const pa_kv_desc &d) {
  const bool fp8 = d.kv_dtype == PA_KV_FP8_E4M3 || d.kv_dtype == PA_KV_FP8_E5M2;
  // automatic choice: the tcgen05 kernel, except 8-bit caches of head_dim 64
  return d.prefill_impl != PA_PREFILL_AUTO ? d.prefill_impl
         : (fp8 && d.head_dim != 128)      ? PA_PREFILL_MMA_SYNC
                                           : PA_PREFILL_TCGEN05;
}

cudaError_t launch_prefill(const pa_kv_desc &d, float *out, float *lse, const void *q,
                           const int32_t *query_start_loc, const void *k_cache,
                           const void *v_cache, const int32_t *block_tables,
                           int32_t max_blocks_per_seq, const int32_t *context_lens,
                           int32_t num_seqs, int32_t max_q_len, float scale, cudaStream_t stream,
                           bool prefix_mode, int num_splits, int split_len, int out_slots) {
  const bool fp8 = d.kv_dtype == PA_KV_FP8_E4M3 || d.kv_dtype == PA_KV_FP8_E5M2;
  const int impl = prefill_impl_of(d);
  if (impl == PA_PREFILL_TCGEN05 || impl == PA_PREFILL_TCGEN05_PAIR)
    return launch_prefill_tc(d, out, lse, q, query_start_loc, k_cache, v_cache, block_tables, max_blocks_per_seq,
                             context_lens, num_seqs, max_q_len, scale, stream, prefix_mode, num_splits, split_len,
                             out_slots, impl == PA_PREFILL_TCGEN05_PAIR);
  const int g = d.num_q_heads / d.num_kv_heads;
  PrefillArgs a;
  a.out = out;
  a.lse = lse;
  a.q = static_cast<const uint16_t *>(q);
  a.query_start_loc = query_start_loc;
  a.k_cache = static_cast<const uint8_t *>(k_cache);
  a.v_cache = static_cast<const uint8_t *>(v_cache);
  a.block_tables = block_tables;
  a.context_lens = context_lens;
  a.max_blocks_per_seq = max_blocks_per_seq;
  a.num_kv_heads = d.num_kv_heads;
  a.num_q_heads = d.num_q_heads;
  a.g = g;
  a.qt = (kPrefillWarps * 16) / g;
  const float ks = (fp8 && d.k_scale != 0.f) ? d.k_scale : 1.f;
  a.qscale = scale * ks * kLog2e;
  a.vscale = (fp8 && d.v_scale != 0.f) ? d.v_scale : 1.f;
  a.qscale0 = scale * kLog2e;
  a.k_scales = fp8 ? d.k_scales : nullptr;
  a.v_scales = fp8 ? d.v_scales : nullptr;
  a.window = d.sliding_window;
  a.chunk = d.attention_chunk;
  a.prefix_mode = prefix_mode ? 1 : 0;
  a.num_splits = prefix_mode ? num_splits : 1;
  a.split_len = split_len;
  a.out_slots = prefix_mode ? out_slots : 1;
  a.err = d.error_word;
  a.checked = d.check_indices;
  a.num_blocks = d.num_blocks;
  void *fn;
  size_t smem;
  if (d.head_dim == 128) {
    fn = d.kv_dtype == PA_KV_FP8_E5M2 ? prefill_fn<128, kKvE5M2>()
         : fp8                         ? prefill_fn<128, kKvFp8>()
         : d.kv_dtype == PA_KV_F16     ? prefill_fn<128, kKvF16>()
                                       : prefill_fn<128, kKvBf16>();
    smem = d.kv_dtype == PA_KV_FP8_E5M2 ? PrefillCfg<128, kKvE5M2, kPrefillWarps>::SMEM
           : fp8                         ? PrefillCfg<128, kKvFp8, kPrefillWarps>::SMEM
                                         : PrefillCfg<128, kKvBf16, kPrefillWarps>::SMEM;
  } else {
    fn = d.kv_dtype == PA_KV_FP8_E5M2 ? prefill_fn<64, kKvE5M2>()
         : fp8                         ? prefill_fn<64, kKvFp8>()
         : d.kv_dtype == PA_KV_F16     ? prefill_fn<64, kKvF16>()
                                       : prefill_fn<64, kKvBf16>();
    smem = d.kv_dtype == PA_KV_FP8_E5M2 ? PrefillCfg<64, kKvE5M2, kPrefillWarps>::SMEM
           : fp8                         ? PrefillCfg<64, kKvFp8, kPrefillWarps>::SMEM
                                         : PrefillCfg<64, kKvBf16, kPrefillWarps>::SMEM;
  }
  if (prepare_kernel(fn, kPrefillWarps * 32, smem) < 1) return cudaErrorInvalidConfiguration;
  const int qtiles = (max_q_len + a.qt - 1) / a.qt;
  if (qtiles == 0 || num_seqs == 0) return cudaSuccess;
  dim3 grid(qtiles, d.num_kv_heads, num_seqs * a.num_splits);
  void *args[] = {&a};
  return cudaLaunchKernel(fn, grid, dim3(kPrefillWarps * 32), args, smem, stream);
}

}  // namespace pa
