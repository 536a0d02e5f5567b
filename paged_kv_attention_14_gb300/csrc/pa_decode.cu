// pa_decode.cu -- split-KV decode attention over the block-paged KV cache.
//
// What it computes: for every sequence s and query head h,
//   out[s][h] = sum_t softmax_t(scale * q[s][h] . K_t) V_t
// over the tokens t < context_lens[s] of kv head h / g, gathered through the
// sequence's block table.  This is the "paged attention (block-paged KV
// cache)" of the vllm.cpp implementation notes ("What's implemented", Model
// forward bullet) over its "Block-Paged KV Cache (FP8/FP16)" (architecture
// figure of "Building and Deploying vllm.cpp ..."), block size 16.  With FP8
// pages ("fp8 halves page size to 1 byte per element", CLI table of the same
// walkthrough) the E4M3 bytes are decoded inside the load and the per-tensor
// scales are folded into the softmax scale (K) and the output (V).
//
// How (GB300 design, not taken from the pages):
//  * Persistent grid, stream-K work split.  The (sequence, kv head, block)
//    list is flattened in sequence-major order and cut into gridDim.x equal
//    contiguous ranges; each CTA owns one range, so a 131072-token sequence
//    next to short ones is balanced to within one block.  A range cuts a
//    (sequence, kv head) segment into at most two pieces per CTA; pieces are
//    written to per-CTA slots and the last CTA to finish a segment (an atomic
//    counter, no waiting) merges them by log-sum-exp in the same launch.
//  * One producer warp streams KV tiles with the TMA engine into an NS-stage
//    shared-memory ring guarded by mbarriers; it prefetches block-table rows
//    32 entries at a time and runs ahead across piece boundaries, so the
//    stream does not stall between sequences.
//  * Two consumers share that framework:
//    - SIMT (group size <= 4): fp32 CUDA-core dot products; 8 lanes share a
//      token row, three xor-shuffles reduce it; tiles arrive by 1-D bulk copy.
//    - MMA (any group size <= 16): per 16-token block, S^T = K Q^T and
//      O^T += V^T P^T as m16n8k16 tensor-core MMAs with the block's tokens as
//      M and the query heads of the group as N (padded to 8 or 16); P^T is
//      produced from the S^T accumulators by an in-register 8x8 transpose
//      (movmatrix).  Tiles arrive by TMA tensor copies with 128B/64B swizzle
//      so every ldmatrix is bank-conflict free.  bf16 KV uses bf16 MMAs with
//      the probabilities split into a bf16 hi + lo pair (near-fp32 accuracy);
//      E4M3 KV is converted exactly to f16 in registers and uses f16 MMAs.
#include <cuda.h>
#include <float.h>
#include <string.h>

#include "pa_device.cuh"
#include "pa_internal.h"

namespace pa {

namespace {

constexpr float kLog2e = 1.4426950408889634f;
constexpr float kLn2 = 0.6931471805599453f;
constexpr int kFlagFirst = 1;
constexpr int kFlagLast = 2;
constexpr int kStageData = 0;
constexpr int kStageEnd = 1;
constexpr int kConsumerWarps = 4;

struct __align__(16) StageHdr {
  long long seg_start;  // flat block index where the (s, kv head) segment starts
  int kind;
  int s;
  int kvh;
  int ntok;    // valid tokens in this stage
  int flags;   // kFlagFirst / kFlagLast of a piece
  int seg_nb;  // blocks of the segment
};

struct DecodeArgs {
  CUtensorMap kmap;  // MMA kernel only: the K cache as [rows = blocks*heads*16][D]
  CUtensorMap vmap;
  float *out;
  float *lse;
  const uint16_t *q;
  const uint8_t *k_cache;
  const uint8_t *v_cache;
  const int32_t *block_tables;
  const int32_t *context_lens;
  int max_blocks_per_seq;
  int num_seqs;
  int num_kv_heads;
  int num_q_heads;
  int g;
  float qscale;  // scale * k_scale * log2(e)
  float vscale;  // v_scale (1 for bf16)
  int32_t *err;
  int32_t *seg_counter;
  float *slot_lse;  // [grid][2][HP], log2 domain
  float *slot_o;    // [grid][2][HP][D]
};

// ---------------------------------------------------------------- workspace

constexpr size_t align256(size_t x) { return (x + 255) & ~size_t(255); }

struct WsLayout {
  size_t counter_off, slot_lse_off, slot_o_off, total;
};

WsLayout ws_layout(int num_seqs, int num_kv_heads, int grid, int hp, int d) {
  WsLayout w;
  w.counter_off = 256;
  w.slot_lse_off = w.counter_off + align256(sizeof(int32_t) * size_t(num_seqs) * num_kv_heads);
  w.slot_o_off = w.slot_lse_off + align256(sizeof(float) * size_t(grid) * 2 * hp);
  w.total = w.slot_o_off + align256(sizeof(float) * size_t(grid) * 2 * hp * d);
  return w;
}

// Output of an empty sequence: zeros and lse = -inf.
__device__ void zero_sequence(const DecodeArgs &a, int s, int D) {
  for (int h = 0; h < a.num_q_heads; ++h) {
    float *o = a.out + (static_cast<int64_t>(s) * a.num_q_heads + h) * D;
    for (int d = 0; d < D; ++d) o[d] = 0.f;
    if (a.lse) a.lse[static_cast<int64_t>(s) * a.num_q_heads + h] = -INFINITY;
  }
}

// --------------------------------------------------------- shared framework

// Pass over context_lens by one warp: the number of 16-token blocks of all
// sequences; empty sequences are zero-filled by the CTA s % gridDim.x.
template <int D>
__device__ long long count_blocks(const DecodeArgs &a, int lane) {
  long long nb_sum = 0;
  const int S = a.num_seqs;
  const int G = gridDim.x;
  for (int base = 0; base < S; base += 256) {
    unsigned acc = 0;
#pragma unroll
    for (int i = 0; i < 8; ++i) {
      const int s = base + i * 32 + lane;
      if (s < S) {
        const int L = __ldg(a.context_lens + s);
        if (L > 0)
          acc += static_cast<unsigned>((L + 15) >> 4);
        else if (s % G == static_cast<int>(blockIdx.x))
          zero_sequence(a, s, D);
      }
    }
    nb_sum += __reduce_add_sync(0xffffffffu, acc);
  }
  return nb_sum;
}

// The producer warp: walks this CTA's range of flat (sequence, kv head,
// block) units and fills the stage ring.  Cfg::issue() starts the copies of
// one block's K and V tiles (one lane per block).
template <class Cfg>
__device__ void produce(const DecodeArgs &a, uint8_t *stages, StageHdr *hdr, uint64_t *full,
                        uint64_t *empty, long long per_cta, long long total, int lane) {
  constexpr int NS = Cfg::NS;
  constexpr int BPS = Cfg::BPS;
  const int S = a.num_seqs;
  const int Hkv = a.num_kv_heads;
  const long long b0 = static_cast<long long>(blockIdx.x) * per_cta;
  const long long b1 = min(b0 + per_cta, total);
  const uint64_t pol = l2_evict_first_policy();
  int stage = 0;
  uint32_t ppar = 1;  // a fresh barrier counts its preceding phase (parity 1) as complete
  bool ok = true;
  int issued = 0;
  if (b0 < b1) {
    // the sequence holding flat block b0, and the flat start of that sequence
    long long pre = 0;
    int s = -1;
    for (int base = 0; base < S && s < 0; base += 32) {
      const int si = base + lane;
      const int L = si < S ? __ldg(a.context_lens + si) : 0;
      const long long v = L > 0 ? static_cast<long long>((L + 15) >> 4) * Hkv : 0;
      long long incl = v;
#pragma unroll
      for (int o = 1; o < 32; o <<= 1) {
        const long long t = __shfl_up_sync(0xffffffffu, incl, o);
        if (lane >= o) incl += t;
      }
      const long long excl = incl - v;
      const bool hit = v > 0 && pre + excl <= b0 && b0 < pre + incl;
      const unsigned m = __ballot_sync(0xffffffffu, hit);
      if (m) {
        const int src = __ffs(m) - 1;
        s = base + src;
        pre += __shfl_sync(0xffffffffu, excl, src);
      } else {
        pre += __shfl_sync(0xffffffffu, incl, 31);
      }
    }
    int L = __ldg(a.context_lens + s);
    int nb = (L + 15) >> 4;
    int kvh = static_cast<int>((b0 - pre) / nb);
    int off = static_cast<int>((b0 - pre) % nb);
    long long cur = b0;
    int win_s = -1, win_base = 0, win_val = 0;
    while (cur < b1 && ok) {
      const long long seg_start = pre + static_cast<long long>(kvh) * nb;
      const long long piece_end = min(b1, seg_start + nb);
      const int npb = static_cast<int>(piece_end - cur);
      for (int k = 0; k < npb; k += BPS) {
        const int nblk = min(BPS, npb - k);
        const int lb0 = off + k;
        if (win_s != s || lb0 < win_base || lb0 + nblk > win_base + 32) {
          win_s = s;
          win_base = lb0;
          const int e = lb0 + lane;
          win_val = e < nb ? __ldg(a.block_tables + static_cast<int64_t>(s) * a.max_blocks_per_seq + e) : 0;
        }
        const int phys = __shfl_sync(0xffffffffu, win_val, (lb0 - win_base + lane) & 31);
        if (!mbar_wait(&empty[stage], ppar)) {
          ok = false;
          break;
        }
        const bool first = (k == 0);
        if (lane == 0) {
          StageHdr h;
          h.seg_start = seg_start;
          h.kind = kStageData;
          h.s = s;
          h.kvh = kvh;
          h.ntok = min(L - lb0 * 16, nblk * 16);
          h.flags = (first ? kFlagFirst : 0) | (k + BPS >= npb ? kFlagLast : 0);
          h.seg_nb = nb;
          hdr[stage] = h;
          const uint32_t bytes = 2u * nblk * Cfg::TILEB + (first ? static_cast<uint32_t>(a.g * Cfg::D * 2) : 0u);
          mbar_arrive_expect_tx(&full[stage], bytes);
        }
        __syncwarp();
        uint8_t *sk = stages + size_t(stage) * Cfg::STAGEB;
        if (lane < nblk) Cfg::issue(a, sk, lane, phys, kvh, &full[stage], pol);
        if (first && lane == 31) {
          const uint16_t *qsrc = a.q + (static_cast<int64_t>(s) * a.num_q_heads + kvh * a.g) * Cfg::D;
          bulk_g2s(sk + Cfg::QOFF, qsrc, static_cast<uint32_t>(a.g * Cfg::D * 2), &full[stage]);
        }
        ++issued;
        if (++stage == NS) {
          stage = 0;
          ppar ^= 1;
        }
      }
      cur = piece_end;
      off = 0;
      if (++kvh == Hkv) {
        kvh = 0;
        pre += static_cast<long long>(nb) * Hkv;
        do {
          ++s;
        } while (s < S && __ldg(a.context_lens + s) <= 0);
        if (s < S) {
          L = __ldg(a.context_lens + s);
          nb = (L + 15) >> 4;
        }
      }
    }
  }
  if (ok) {
    if (mbar_wait(&empty[stage], ppar)) {
      if (lane == 0) {
        hdr[stage].kind = kStageEnd;
        mbar_arrive(&full[stage]);
      }
    } else {
      ok = false;
    }
  }
  if (!ok) {
    if (lane == 0) atomicOr(a.err, kErrWaitTimeout);
    // let the copies already issued land before the CTA can exit
    for (int i = 1; i <= min(issued, NS); ++i) {
      int st = stage - i;
      uint32_t par = ppar ^ 1;
      if (st < 0) {
        st += NS;
        par ^= 1;
      }
      mbar_wait(&full[st], par);
    }
  }
}

// Finish one piece.  Each consumer warp w has left in red[w] its partial
// state for every head j of the group: unnormalised O[j][0..D), the running
// max m (log2 domain) at [D] and the sum l at [D+1] (head stride D + 2,
// HP heads per warp).  Combines the warps, then writes the output (whole
// segment in this CTA) or this CTA's slot, and the last CTA of a split
// segment merges all slots of that segment.
template <int D, int HP, int NC>
__device__ void finish_piece(const DecodeArgs &a, const StageHdr &h, const float *red, long long per_cta,
                             int *s_flag, int tid) {
  constexpr int CT = NC * 32;
  constexpr int REDW = HP * (D + 2);
  const long long c1 = h.seg_start / per_cta;
  const long long c2 = (h.seg_start + h.seg_nb - 1) / per_cta;
  const bool split = c1 != c2;
  const int me = blockIdx.x;
  const int my_slot = (h.seg_start <= static_cast<long long>(me) * per_cta) ? 0 : 1;
  const int hq0 = h.kvh * a.g;
  for (int idx = tid; idx < a.g * D; idx += CT) {
    const int j = idx / D;
    const int d = idx - j * D;
    float M = -INFINITY;
#pragma unroll
    for (int w = 0; w < NC; ++w) M = fmaxf(M, red[w * REDW + j * (D + 2) + D]);
    float Ls = 0.f, O = 0.f;
#pragma unroll
    for (int w = 0; w < NC; ++w) {
      const float mw = red[w * REDW + j * (D + 2) + D];
      if (mw != -INFINITY) {
        const float c = exp2f(mw - M);
        Ls += red[w * REDW + j * (D + 2) + D + 1] * c;
        O += red[w * REDW + j * (D + 2) + d] * c;
      }
    }
    const float res = O / Ls;
    const float lse2 = M + log2f(Ls);
    if (!split) {
      a.out[(static_cast<int64_t>(h.s) * a.num_q_heads + hq0 + j) * D + d] = res * a.vscale;
      if (a.lse && d == 0) a.lse[static_cast<int64_t>(h.s) * a.num_q_heads + hq0 + j] = lse2 * kLn2;
    } else {
      const int64_t sl = (static_cast<int64_t>(me) * 2 + my_slot) * HP + j;
      a.slot_o[sl * D + d] = res;
      if (d == 0) a.slot_lse[sl] = lse2;
    }
  }
  if (split) {
    __threadfence();
    named_bar_sync(1, CT);
    if (tid == 0) {
      const int seg = h.s * a.num_kv_heads + h.kvh;
      const int npieces = static_cast<int>(c2 - c1 + 1);
      const int prev = atomicAdd(a.seg_counter + seg, 1);
      const int last = prev == npieces - 1;
      if (last) {
        a.seg_counter[seg] = 0;  // ready for the next launch
        __threadfence();
      }
      *s_flag = last;
    }
    named_bar_sync(1, CT);
    if (*s_flag) {
      for (int idx = tid; idx < a.g * D; idx += CT) {
        const int j = idx / D;
        const int d = idx - j * D;
        float M = -INFINITY;
        for (long long c = c1; c <= c2; ++c) {
          const int sl = (h.seg_start <= c * per_cta) ? 0 : 1;
          M = fmaxf(M, __ldcg(a.slot_lse + (c * 2 + sl) * HP + j));
        }
        float W = 0.f, O = 0.f;
        for (long long c = c1; c <= c2; ++c) {
          const int sl = (h.seg_start <= c * per_cta) ? 0 : 1;
          const int64_t base = (c * 2 + sl) * HP + j;
          const float w = exp2f(__ldcg(a.slot_lse + base) - M);
          W += w;
          O += w * __ldcg(a.slot_o + base * D + d);
        }
        a.out[(static_cast<int64_t>(h.s) * a.num_q_heads + hq0 + j) * D + d] = O / W * a.vscale;
        if (a.lse && d == 0) a.lse[static_cast<int64_t>(h.s) * a.num_q_heads + hq0 + j] = (M + log2f(W)) * kLn2;
      }
    }
  }
  named_bar_sync(1, CT);  // the reduction buffer is free again
}

// Kernel prologue shared by both consumers: barrier init, block count,
// per-CTA range.  Returns per_cta and (for the producer warp) the total.
template <class Cfg>
__device__ long long prologue(const DecodeArgs &a, uint64_t *full, uint64_t *empty, long long *total_out,
                              long long *s_per_cta) {
  const int tid = threadIdx.x;
  const int warp = tid >> 5;
  if (tid == 0) {
    for (int st = 0; st < Cfg::NS; ++st) {
      mbar_init(&full[st], 1);
      mbar_init(&empty[st], Cfg::NC);
    }
    fence_mbar_init();
  }
  if (warp == Cfg::NC) {
    const long long nb_sum = count_blocks<Cfg::D>(a, tid & 31);
    *total_out = nb_sum * a.num_kv_heads;
    if ((tid & 31) == 0) *s_per_cta = (*total_out + gridDim.x - 1) / gridDim.x;
  }
  __syncthreads();
  return *s_per_cta;
}

// ============================================================ SIMT consumer

// Which head_dim elements lane j8 (0..7) of an 8-lane token group holds, and
// how it loads them from a cached row.  bf16 rows: 16-byte chunks j8,
// j8 + 8, ... (each quarter-warp reads one contiguous 128-byte span).  E4M3
// rows: one contiguous run of D/8 bytes per lane.
template <int D, int KVT>
struct RowSlice {
  static constexpr int EPL = D / 8;
  __device__ static __forceinline__ int dim(int j8, int e) {
    if (KVT == kKvBf16) return ((e >> 3) * 8 + j8) * 8 + (e & 7);
    return j8 * EPL + e;
  }
  __device__ static __forceinline__ void load(const uint8_t *row, int j8, float (&x)[EPL]) {
    if (KVT == kKvBf16) {
#pragma unroll
      for (int c = 0; c < EPL / 8; ++c) {
        const uint4 u = *reinterpret_cast<const uint4 *>(row + (c * 8 + j8) * 16);
        x[c * 8 + 0] = bf16lo(u.x);
        x[c * 8 + 1] = bf16hi(u.x);
        x[c * 8 + 2] = bf16lo(u.y);
        x[c * 8 + 3] = bf16hi(u.y);
        x[c * 8 + 4] = bf16lo(u.z);
        x[c * 8 + 5] = bf16hi(u.z);
        x[c * 8 + 6] = bf16lo(u.w);
        x[c * 8 + 7] = bf16hi(u.w);
      }
    } else if (EPL == 16) {
      const uint4 u = *reinterpret_cast<const uint4 *>(row + j8 * 16);
      const uint32_t w[4] = {u.x, u.y, u.z, u.w};
#pragma unroll
      for (int c = 0; c < 4; ++c) {
        e4m3x2_to_f32(static_cast<uint16_t>(w[c] & 0xffffu), x[4 * c + 0], x[4 * c + 1]);
        e4m3x2_to_f32(static_cast<uint16_t>(w[c] >> 16), x[4 * c + 2], x[4 * c + 3]);
      }
    } else {
      const uint2 u = *reinterpret_cast<const uint2 *>(row + j8 * 8);
      const uint32_t w[2] = {u.x, u.y};
#pragma unroll
      for (int c = 0; c < 2; ++c) {
        e4m3x2_to_f32(static_cast<uint16_t>(w[c] & 0xffffu), x[4 * c + 0], x[4 * c + 1]);
        e4m3x2_to_f32(static_cast<uint16_t>(w[c] >> 16), x[4 * c + 2], x[4 * c + 3]);
      }
    }
  }
};

template <int D_, int KVT, int GP_, int BPS_, int NS_>
struct SimtCfg {
  static constexpr int D = D_;
  static constexpr int GP = GP_;
  static constexpr int HP = GP_;  // heads per warp in the reduction buffer
  static constexpr int BPS = BPS_;
  static constexpr int NS = NS_;
  static constexpr int NC = kConsumerWarps;
  static constexpr int ESZ = (KVT == kKvBf16) ? 2 : 1;
  static constexpr int ROWB = D * ESZ;
  static constexpr int TILEB = 16 * ROWB;       // one (block, kv head) tile
  static constexpr int KVB = BPS * TILEB;       // K (or V) bytes of a stage
  static constexpr int QB = ((GP * D * 2 + 127) / 128) * 128;
  static constexpr int QOFF = 2 * KVB;
  static constexpr int STAGEB = 2 * KVB + QB;
  static constexpr int EPL = D / 8;
  static constexpr int NG = NC * 4;             // 8-lane token groups
  static constexpr int TPG = BPS * 16 / NG;     // tokens per group per stage
  static constexpr int NTHREADS = (NC + 1) * 32;
  static constexpr int REDW = HP * (D + 2);
  static constexpr size_t SMEM = size_t(NS) * STAGEB + NS * sizeof(StageHdr) + 2 * NS * sizeof(uint64_t) +
                                 size_t(NC) * REDW * sizeof(float) + 16;
  static_assert(TPG >= 1 && TPG * NG == BPS * 16, "stage must split evenly over groups");
  static_assert(BPS <= 31, "one producer lane per block plus one for q");

  __device__ static __forceinline__ void issue(const DecodeArgs &a, uint8_t *sk, int i, int phys, int kvh,
                                               uint64_t *bar, uint64_t pol) {
    const int64_t tile = (static_cast<int64_t>(phys) * a.num_kv_heads + kvh) * TILEB;
    bulk_g2s(sk + i * TILEB, a.k_cache + tile, TILEB, bar, pol);
    bulk_g2s(sk + KVB + i * TILEB, a.v_cache + tile, TILEB, bar, pol);
  }
};

template <int D, int KVT, int GP, int BPS, int NS>
__global__ void __launch_bounds__((kConsumerWarps + 1) * 32, 2) decode_simt_kernel(const __grid_constant__ DecodeArgs a) {
  using C = SimtCfg<D, KVT, GP, BPS, NS>;
  using RS = RowSlice<D, KVT>;
  constexpr int EPL = C::EPL;
  constexpr int NC = C::NC;
  extern __shared__ __align__(128) uint8_t smem[];
  uint8_t *stages = smem;
  StageHdr *hdr = reinterpret_cast<StageHdr *>(smem + size_t(NS) * C::STAGEB);
  uint64_t *full = reinterpret_cast<uint64_t *>(hdr + NS);
  uint64_t *empty = full + NS;
  float *red = reinterpret_cast<float *>(empty + NS);
  __shared__ long long s_per_cta;
  __shared__ int s_flag;

  const int tid = threadIdx.x;
  const int warp = tid >> 5;
  const int lane = tid & 31;
  long long total = 0;
  const long long per_cta = prologue<C>(a, full, empty, &total, &s_per_cta);
  if (warp == NC) {
    produce<C>(a, stages, hdr, full, empty, per_cta, total, lane);
    return;
  }

  const int gid = warp * 4 + (lane >> 3);
  const int j8 = lane & 7;
  float q[GP][EPL], o[GP][EPL], m[GP], l[GP];
#pragma unroll
  for (int j = 0; j < GP; ++j) {
    m[j] = -INFINITY;
    l[j] = 0.f;
#pragma unroll
    for (int e = 0; e < EPL; ++e) {
      q[j][e] = 0.f;
      o[j][e] = 0.f;
    }
  }
  int stage = 0;
  uint32_t cpar = 0;
  for (;;) {
    if (!mbar_wait(&full[stage], cpar)) {
      if (lane == 0) atomicOr(a.err, kErrWaitTimeout);
      break;
    }
    const StageHdr h = hdr[stage];
    if (h.kind == kStageEnd) break;
    const uint8_t *Ks = stages + size_t(stage) * C::STAGEB;
    const uint8_t *Vs = Ks + C::KVB;
    if (h.flags & kFlagFirst) {
      const uint16_t *Qs = reinterpret_cast<const uint16_t *>(Ks + C::QOFF);
#pragma unroll
      for (int j = 0; j < GP; ++j) {
        m[j] = -INFINITY;
        l[j] = 0.f;
#pragma unroll
        for (int e = 0; e < EPL; ++e) {
          q[j][e] = j < a.g ? __uint_as_float(static_cast<uint32_t>(Qs[j * D + RS::dim(j8, e)]) << 16) * a.qscale : 0.f;
          o[j][e] = 0.f;
        }
      }
    }
    float x[C::TPG][GP];
#pragma unroll
    for (int i = 0; i < C::TPG; ++i) {
      const int r = gid + C::NG * i;
      const bool valid = r < h.ntok;
      float acc[GP];
#pragma unroll
      for (int j = 0; j < GP; ++j) acc[j] = 0.f;
      if (valid) {
        float kv[EPL];
        RS::load(Ks + (r >> 4) * C::TILEB + (r & 15) * C::ROWB, j8, kv);
#pragma unroll
        for (int j = 0; j < GP; ++j)
#pragma unroll
          for (int e = 0; e < EPL; ++e) acc[j] = fmaf(q[j][e], kv[e], acc[j]);
      }
#pragma unroll
      for (int j = 0; j < GP; ++j) {
        acc[j] += __shfl_xor_sync(0xffffffffu, acc[j], 1);
        acc[j] += __shfl_xor_sync(0xffffffffu, acc[j], 2);
        acc[j] += __shfl_xor_sync(0xffffffffu, acc[j], 4);
        x[i][j] = valid ? acc[j] : -INFINITY;
      }
    }
#pragma unroll
    for (int j = 0; j < GP; ++j) {
      float mx = m[j];
#pragma unroll
      for (int i = 0; i < C::TPG; ++i) mx = fmaxf(mx, x[i][j]);
      if (mx > m[j]) {
        const float c = exp2f(m[j] - mx);
        l[j] *= c;
#pragma unroll
        for (int e = 0; e < EPL; ++e) o[j][e] *= c;
        m[j] = mx;
      }
#pragma unroll
      for (int i = 0; i < C::TPG; ++i) {
        x[i][j] = (x[i][j] == -INFINITY) ? 0.f : exp2f(x[i][j] - m[j]);
        l[j] += x[i][j];
      }
    }
#pragma unroll
    for (int i = 0; i < C::TPG; ++i) {
      const int r = gid + C::NG * i;
      if (r < h.ntok) {
        float kv[EPL];
        RS::load(Vs + (r >> 4) * C::TILEB + (r & 15) * C::ROWB, j8, kv);
#pragma unroll
        for (int j = 0; j < GP; ++j)
#pragma unroll
          for (int e = 0; e < EPL; ++e) o[j][e] = fmaf(x[i][j], kv[e], o[j][e]);
      }
    }
    __syncwarp();
    if (lane == 0) mbar_arrive(&empty[stage]);
    if (++stage == NS) {
      stage = 0;
      cpar ^= 1;
    }
    if (!(h.flags & kFlagLast)) continue;

    // combine the four token groups of this warp, then hand over to the CTA
#pragma unroll
    for (int sh = 8; sh <= 16; sh <<= 1) {
#pragma unroll
      for (int j = 0; j < GP; ++j) {
        const float mo = __shfl_xor_sync(0xffffffffu, m[j], sh);
        const float lo = __shfl_xor_sync(0xffffffffu, l[j], sh);
        const float mn = fmaxf(m[j], mo);
        const float ca = (m[j] == -INFINITY) ? 0.f : exp2f(m[j] - mn);
        const float cb = (mo == -INFINITY) ? 0.f : exp2f(mo - mn);
        l[j] = l[j] * ca + lo * cb;
#pragma unroll
        for (int e = 0; e < EPL; ++e) o[j][e] = o[j][e] * ca + __shfl_xor_sync(0xffffffffu, o[j][e], sh) * cb;
        m[j] = mn;
      }
    }
    float *rw = red + warp * C::REDW;
    if (lane < 8) {
#pragma unroll
      for (int j = 0; j < GP; ++j) {
#pragma unroll
        for (int e = 0; e < EPL; ++e) rw[j * (D + 2) + RS::dim(lane, e)] = o[j][e];
        if (lane == 0) {
          rw[j * (D + 2) + D] = m[j];
          rw[j * (D + 2) + D + 1] = l[j];
        }
      }
    }
    named_bar_sync(1, NC * 32);
    finish_piece<D, C::HP, NC>(a, h, red, per_cta, &s_flag, tid);
  }
}

// ============================================================= MMA consumer

// Byte offset of 16-byte chunk `ch` of token row `t` in a tile stored by TMA
// with 128-byte (rows of 128 B) or 64-byte (rows of 64 B) swizzling.  Wider
// rows are split into 128-byte boxes of 16 rows each.
template <int ROWB>
__device__ __forceinline__ uint32_t swz_off(int t, int ch) {
  if constexpr (ROWB >= 128) {
    const int box = ch >> 3;
    const int c = ch & 7;
    return static_cast<uint32_t>(box * 2048 + t * 128 + ((c ^ (t & 7)) << 4));
  } else {
    return static_cast<uint32_t>(t * 64 + ((ch ^ ((t >> 1) & 3)) << 4));
  }
}

template <int D_, int KVT_, int NN_, int BPS_, int NS_>
struct MmaCfg {
  static constexpr int D = D_;
  static constexpr int KVT = KVT_;
  static constexpr int NN = NN_;           // n-tiles of 8 query heads
  static constexpr int HP = 8 * NN_;       // heads per warp in the reduction buffer
  static constexpr int BPS = BPS_;
  static constexpr int NS = NS_;
  static constexpr int NC = kConsumerWarps;
  static constexpr int ESZ = (KVT == kKvBf16) ? 2 : 1;
  static constexpr int ROWB = D * ESZ;
  static constexpr int BOXB = ROWB >= 128 ? 128 : ROWB;   // bytes of a box row
  static constexpr int NBOX = ROWB / BOXB;
  static constexpr int BOXCOLS = BOXB / ESZ;
  static constexpr int TILEB = 16 * ROWB;
  static constexpr int KVB = BPS * TILEB;
  static constexpr int QB = ((HP * D * 2 + 1023) / 1024) * 1024;
  static constexpr int QOFF = 2 * KVB;
  static constexpr int STAGEB = 2 * KVB + QB;
  static constexpr int BPW = BPS / NC;     // blocks per consumer warp per stage
  static constexpr int NTHREADS = (NC + 1) * 32;
  static constexpr int REDW = HP * (D + 2);
  static constexpr size_t SMEM = 1024 + size_t(NS) * STAGEB + NS * sizeof(StageHdr) +
                                 2 * NS * sizeof(uint64_t) + size_t(NC) * REDW * sizeof(float) + 16;
  static_assert(BPS % NC == 0, "blocks of a stage split evenly over consumer warps");
  static_assert(TILEB % 1024 == 0 || ROWB == 64, "tiles keep the swizzle alignment");

  __device__ static __forceinline__ void issue(const DecodeArgs &a, uint8_t *sk, int i, int phys, int kvh,
                                               uint64_t *bar, uint64_t pol) {
    const int row = (phys * a.num_kv_heads + kvh) * 16;
#pragma unroll
    for (int b = 0; b < NBOX; ++b) {
      tma_load_2d(sk + i * TILEB + b * 16 * BOXB, &a.kmap, b * BOXCOLS, row, bar, pol);
      tma_load_2d(sk + KVB + i * TILEB + b * 16 * BOXB, &a.vmap, b * BOXCOLS, row, bar, pol);
    }
  }
};

template <int D, int KVT, int NN, int BPS, int NS>
__global__ void __launch_bounds__((kConsumerWarps + 1) * 32, 1) decode_mma_kernel(const __grid_constant__ DecodeArgs a) {
  using C = MmaCfg<D, KVT, NN, BPS, NS>;
  constexpr int NC = C::NC;
  constexpr int MT = D / 16;  // m-tiles of O^T (16 head_dim rows each) = k-steps of S^T
  extern __shared__ uint8_t smem_raw[];
  uint8_t *smem = reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint8_t *stages = smem;
  StageHdr *hdr = reinterpret_cast<StageHdr *>(smem + size_t(NS) * C::STAGEB);
  uint64_t *full = reinterpret_cast<uint64_t *>(hdr + NS);
  uint64_t *empty = full + NS;
  float *red = reinterpret_cast<float *>(empty + NS);
  __shared__ long long s_per_cta;
  __shared__ int s_flag;

  const int tid = threadIdx.x;
  const int warp = tid >> 5;
  const int lane = tid & 31;
  long long total = 0;
  const long long per_cta = prologue<C>(a, full, empty, &total, &s_per_cta);
  if (warp == NC) {
    produce<C>(a, stages, hdr, full, empty, per_cta, total, lane);
    return;
  }

  const int r = lane >> 2;  // fragment row group
  const int c = lane & 3;   // fragment column pair
  const int lm = lane >> 3;  // ldmatrix: which 8x8 matrix this lane addresses
  const int lr = lane & 7;   // ldmatrix: which row of it
  uint32_t qb[MT][NN][2];    // Q^T B fragments (bf16 or f16 pairs)
  float oacc[MT][NN][4];     // O^T accumulators
  float m[NN][2], l[NN][2];  // per head 2c, 2c+1 of each n-tile
#pragma unroll
  for (int nn = 0; nn < NN; ++nn) {
    m[nn][0] = m[nn][1] = -INFINITY;
    l[nn][0] = l[nn][1] = 0.f;
  }
  int stage = 0;
  uint32_t cpar = 0;
  for (;;) {
    if (!mbar_wait(&full[stage], cpar)) {
      if (lane == 0) atomicOr(a.err, kErrWaitTimeout);
      break;
    }
    const StageHdr h = hdr[stage];
    if (h.kind == kStageEnd) break;
    const uint8_t *Ks = stages + size_t(stage) * C::STAGEB;
    const uint8_t *Vs = Ks + C::KVB;
    if (h.flags & kFlagFirst) {
      // Q^T fragments of this piece's query heads (zero past g)
      const uint16_t *Qs = reinterpret_cast<const uint16_t *>(Ks + C::QOFF);
#pragma unroll
      for (int nn = 0; nn < NN; ++nn) {
        const int n = nn * 8 + r;
        const bool hv = n < a.g;
#pragma unroll
        for (int ks = 0; ks < MT; ++ks) {
          if (KVT == kKvBf16) {
            // k = 2c, 2c+1 <-> d = 16ks + 2c + {0,1};  k + 8 <-> d + 8
            const int d0 = ks * 16 + 2 * c;
            qb[ks][nn][0] = hv ? *reinterpret_cast<const uint32_t *>(Qs + n * D + d0) : 0u;
            qb[ks][nn][1] = hv ? *reinterpret_cast<const uint32_t *>(Qs + n * D + d0 + 8) : 0u;
          } else {
            // k = 2c, 2c+1 <-> d = 16ks + 4c + {0,1};  k + 8 <-> d = 16ks + 4c + {2,3}
            const int d0 = ks * 16 + 4 * c;
            uint32_t w0 = 0, w1 = 0;
            if (hv) {
              w0 = *reinterpret_cast<const uint32_t *>(Qs + n * D + d0);
              w1 = *reinterpret_cast<const uint32_t *>(Qs + n * D + d0 + 2);
            }
            qb[ks][nn][0] = pack_f16x2(bf16lo(w0), bf16hi(w0));
            qb[ks][nn][1] = pack_f16x2(bf16lo(w1), bf16hi(w1));
          }
        }
        m[nn][0] = m[nn][1] = -INFINITY;
        l[nn][0] = l[nn][1] = 0.f;
#pragma unroll
        for (int mt = 0; mt < MT; ++mt) oacc[mt][nn][0] = oacc[mt][nn][1] = oacc[mt][nn][2] = oacc[mt][nn][3] = 0.f;
      }
    }
#pragma unroll
    for (int bw = 0; bw < C::BPW; ++bw) {
      const int bi = warp + NC * bw;  // block of the stage
      const int vt = h.ntok - 16 * bi;  // valid tokens of this block (<= 0: none)
      if (vt <= 0) break;
      const uint32_t kt = smem_u32(Ks + bi * C::TILEB);
      const uint32_t vtl = smem_u32(Vs + bi * C::TILEB);
      // ---- S^T (16 tokens x 8 heads per n-tile) = K Q^T
      float sacc[NN][4];
#pragma unroll
      for (int nn = 0; nn < NN; ++nn) sacc[nn][0] = sacc[nn][1] = sacc[nn][2] = sacc[nn][3] = 0.f;
      if (KVT == kKvBf16) {
#pragma unroll
        for (int ks = 0; ks < MT; ++ks) {
          uint32_t a0, a1, a2, a3;
          ldmatrix_x4(a0, a1, a2, a3, kt + swz_off<C::ROWB>(lr + (lm & 1) * 8, 2 * ks + (lm >> 1)));
#pragma unroll
          for (int nn = 0; nn < NN; ++nn) mma_bf16_16816(sacc[nn], a0, a1, a2, a3, qb[ks][nn][0], qb[ks][nn][1]);
        }
      } else {
#pragma unroll
        for (int j = 0; j < MT; j += 2) {
          uint32_t r0, r1, r2, r3;
          ldmatrix_x4(r0, r1, r2, r3, kt + swz_off<C::ROWB>(lr + (lm & 1) * 8, j + (lm >> 1)));
          const uint32_t a0 = e4m3x2_to_f16x2(static_cast<uint16_t>(r0 & 0xffffu));
          const uint32_t a2 = e4m3x2_to_f16x2(static_cast<uint16_t>(r0 >> 16));
          const uint32_t a1 = e4m3x2_to_f16x2(static_cast<uint16_t>(r1 & 0xffffu));
          const uint32_t a3 = e4m3x2_to_f16x2(static_cast<uint16_t>(r1 >> 16));
#pragma unroll
          for (int nn = 0; nn < NN; ++nn) mma_f16_16816(sacc[nn], a0, a1, a2, a3, qb[j][nn][0], qb[j][nn][1]);
          const uint32_t b0 = e4m3x2_to_f16x2(static_cast<uint16_t>(r2 & 0xffffu));
          const uint32_t b2 = e4m3x2_to_f16x2(static_cast<uint16_t>(r2 >> 16));
          const uint32_t b1 = e4m3x2_to_f16x2(static_cast<uint16_t>(r3 & 0xffffu));
          const uint32_t b3 = e4m3x2_to_f16x2(static_cast<uint16_t>(r3 >> 16));
#pragma unroll
          for (int nn = 0; nn < NN; ++nn) mma_f16_16816(sacc[nn], b0, b1, b2, b3, qb[j + 1][nn][0], qb[j + 1][nn][1]);
        }
      }
      // ---- online softmax over the block's tokens, per head (column)
      uint32_t pb[NN][2], pbl[NN][2];
      const bool v_lo = r < vt, v_hi = r + 8 < vt;
#pragma unroll
      for (int nn = 0; nn < NN; ++nn) {
        float s0 = v_lo ? sacc[nn][0] * a.qscale : -INFINITY;
        float s1 = v_lo ? sacc[nn][1] * a.qscale : -INFINITY;
        float s2 = v_hi ? sacc[nn][2] * a.qscale : -INFINITY;
        float s3 = v_hi ? sacc[nn][3] * a.qscale : -INFINITY;
        float c0 = fmaxf(s0, s2), c1 = fmaxf(s1, s3);
#pragma unroll
        for (int o = 4; o < 32; o <<= 1) {
          c0 = fmaxf(c0, __shfl_xor_sync(0xffffffffu, c0, o));
          c1 = fmaxf(c1, __shfl_xor_sync(0xffffffffu, c1, o));
        }
        const float mn0 = fmaxf(m[nn][0], c0), mn1 = fmaxf(m[nn][1], c1);  // finite: vt >= 1
        const float k0 = exp2f(m[nn][0] - mn0), k1 = exp2f(m[nn][1] - mn1);
        m[nn][0] = mn0;
        m[nn][1] = mn1;
        const float p0 = exp2f(s0 - mn0), p1 = exp2f(s1 - mn1);
        const float p2 = exp2f(s2 - mn0), p3 = exp2f(s3 - mn1);
        l[nn][0] = l[nn][0] * k0 + p0 + p2;
        l[nn][1] = l[nn][1] * k1 + p1 + p3;
#pragma unroll
        for (int mt = 0; mt < MT; ++mt) {
          oacc[mt][nn][0] *= k0;
          oacc[mt][nn][2] *= k0;
          oacc[mt][nn][1] *= k1;
          oacc[mt][nn][3] *= k1;
        }
        if (KVT == kKvBf16) {
          const uint32_t h01 = pack_bf16x2(p0, p1), h23 = pack_bf16x2(p2, p3);
          pb[nn][0] = movmatrix_trans(h01);
          pb[nn][1] = movmatrix_trans(h23);
          pbl[nn][0] = movmatrix_trans(pack_bf16x2(p0 - bf16lo(h01), p1 - bf16hi(h01)));
          pbl[nn][1] = movmatrix_trans(pack_bf16x2(p2 - bf16lo(h23), p3 - bf16hi(h23)));
        } else {
          pb[nn][0] = movmatrix_trans(pack_f16x2(p0, p1));
          pb[nn][1] = movmatrix_trans(pack_f16x2(p2, p3));
        }
      }
      // ---- O^T += V^T P^T
      // Tokens past the block's valid count may hold anything (NaN included);
      // a zero probability does not cancel them (0 * NaN = NaN), so their
      // V^T fragment entries are zeroed: mk_lo covers tokens 2c, 2c+1 and
      // mk_hi tokens 2c+8, 2c+9 of this lane.
      const uint32_t mk_lo = (2 * c < vt ? 0x0000ffffu : 0u) | (2 * c + 1 < vt ? 0xffff0000u : 0u);
      const uint32_t mk_hi = (2 * c + 8 < vt ? 0x0000ffffu : 0u) | (2 * c + 9 < vt ? 0xffff0000u : 0u);
      if (KVT == kKvBf16) {
#pragma unroll
        for (int mt = 0; mt < MT; ++mt) {
          uint32_t a0, a1, a2, a3;
          ldmatrix_x4_trans(a0, a1, a2, a3, vtl + swz_off<C::ROWB>(lr + (lm >> 1) * 8, 2 * mt + (lm & 1)));
          a0 &= mk_lo;
          a1 &= mk_lo;
          a2 &= mk_hi;
          a3 &= mk_hi;
#pragma unroll
          for (int nn = 0; nn < NN; ++nn) {
            mma_bf16_16816(oacc[mt][nn], a0, a1, a2, a3, pb[nn][0], pb[nn][1]);
            mma_bf16_16816(oacc[mt][nn], a0, a1, a2, a3, pbl[nn][0], pbl[nn][1]);
          }
        }
      } else {
#pragma unroll
        for (int j = 0; j < MT; j += 2) {
          uint32_t r0, r1, r2, r3;
          ldmatrix_x4_trans(r0, r1, r2, r3, vtl + swz_off<C::ROWB>(lr + (lm & 1) * 8, j + (lm >> 1)));
          // r0: tokens 2c, 2c+1 (of 0-7) x d = 16j + 2r, 2r+1 as bytes (t,d),(t,d+1),(t+1,d),(t+1,d+1)
          const uint32_t x0 = __byte_perm(r0, 0, 0x3120), x1 = __byte_perm(r1, 0, 0x3120);
          const uint32_t y0 = __byte_perm(r2, 0, 0x3120), y1 = __byte_perm(r3, 0, 0x3120);
          const uint32_t a0 = e4m3x2_to_f16x2(static_cast<uint16_t>(x0 & 0xffffu)) & mk_lo;
          const uint32_t a1 = e4m3x2_to_f16x2(static_cast<uint16_t>(x0 >> 16)) & mk_lo;
          const uint32_t a2 = e4m3x2_to_f16x2(static_cast<uint16_t>(x1 & 0xffffu)) & mk_hi;
          const uint32_t a3 = e4m3x2_to_f16x2(static_cast<uint16_t>(x1 >> 16)) & mk_hi;
          const uint32_t b0 = e4m3x2_to_f16x2(static_cast<uint16_t>(y0 & 0xffffu)) & mk_lo;
          const uint32_t b1 = e4m3x2_to_f16x2(static_cast<uint16_t>(y0 >> 16)) & mk_lo;
          const uint32_t b2 = e4m3x2_to_f16x2(static_cast<uint16_t>(y1 & 0xffffu)) & mk_hi;
          const uint32_t b3 = e4m3x2_to_f16x2(static_cast<uint16_t>(y1 >> 16)) & mk_hi;
#pragma unroll
          for (int nn = 0; nn < NN; ++nn) {
            mma_f16_16816(oacc[j][nn], a0, a1, a2, a3, pb[nn][0], pb[nn][1]);
            mma_f16_16816(oacc[j + 1][nn], b0, b1, b2, b3, pb[nn][0], pb[nn][1]);
          }
        }
      }
    }
    __syncwarp();
    if (lane == 0) mbar_arrive(&empty[stage]);
    if (++stage == NS) {
      stage = 0;
      cpar ^= 1;
    }
    if (!(h.flags & kFlagLast)) continue;

    // ---- this warp's partial state to the reduction buffer
#pragma unroll
    for (int nn = 0; nn < NN; ++nn)
#pragma unroll
      for (int e = 0; e < 2; ++e)
#pragma unroll
        for (int o = 4; o < 32; o <<= 1) l[nn][e] += __shfl_xor_sync(0xffffffffu, l[nn][e], o);
    float *rw = red + warp * C::REDW;
#pragma unroll
    for (int nn = 0; nn < NN; ++nn) {
      const int h0 = nn * 8 + 2 * c;
      if (r == 0) {
        rw[h0 * (D + 2) + D] = m[nn][0];
        rw[h0 * (D + 2) + D + 1] = l[nn][0];
        rw[(h0 + 1) * (D + 2) + D] = m[nn][1];
        rw[(h0 + 1) * (D + 2) + D + 1] = l[nn][1];
      }
#pragma unroll
      for (int mt = 0; mt < MT; ++mt) {
        // bf16: rows r, r+8 of m-tile mt are d = 16mt + r, 16mt + 8 + r;
        // E4M3: d = 16mt + 2r, 16mt + 2r + 1
        const int dlo = (KVT == kKvBf16) ? mt * 16 + r : mt * 16 + 2 * r;
        const int dhi = (KVT == kKvBf16) ? dlo + 8 : dlo + 1;
        rw[h0 * (D + 2) + dlo] = oacc[mt][nn][0];
        rw[(h0 + 1) * (D + 2) + dlo] = oacc[mt][nn][1];
        rw[h0 * (D + 2) + dhi] = oacc[mt][nn][2];
        rw[(h0 + 1) * (D + 2) + dhi] = oacc[mt][nn][3];
      }
    }
    named_bar_sync(1, NC * 32);
    finish_piece<D, C::HP, NC>(a, h, red, per_cta, &s_flag, tid);
  }
}

// -------------------------------------------------------------- dispatch

struct DeviceInfo {
  int sm_count = 0;
};

DeviceInfo &device_info() {
  static DeviceInfo info[64];
  int dev = 0;
  cudaGetDevice(&dev);
  DeviceInfo &d = info[dev & 63];
  if (d.sm_count == 0) {
    int n = 0;
    cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev);
    d.sm_count = n > 0 ? n : 1;
  }
  return d;
}

struct KernelInfo {
  void *fn = nullptr;
  size_t smem = 0;
  int threads = 0;
  int hp = 0;  // heads per slot
  bool mma = false;
  int box_cols = 0;  // MMA: columns of a TMA box
  int swizzle = 0;   // MMA: 128 or 64
};

template <class Cfg, class Fn>
KernelInfo info_of(Fn fn, bool mma) {
  KernelInfo k;
  k.fn = reinterpret_cast<void *>(fn);
  k.smem = Cfg::SMEM;
  k.threads = Cfg::NTHREADS;
  k.hp = Cfg::HP;
  k.mma = mma;
  return k;
}

// SIMT: stages of about 32 KB, three of them, two CTAs per SM
template <int D, int KVT, int GP>
KernelInfo simt_info() {
  constexpr int ESZ = KVT == kKvBf16 ? 2 : 1;
  constexpr int BPS = (D * ESZ >= 256) ? 4 : 8;
  using Cfg = SimtCfg<D, KVT, GP, BPS, 3>;
  return info_of<Cfg>(&decode_simt_kernel<D, KVT, GP, BPS, 3>, false);
}

// MMA: 4 blocks per stage, about 128 KB of stages, one CTA per SM
template <int D, int KVT, int NN>
KernelInfo mma_info() {
  constexpr int ESZ = KVT == kKvBf16 ? 2 : 1;
  constexpr int TILEB = 16 * D * ESZ;
  constexpr int NS = (131072 / (8 * TILEB)) < 2 ? 2 : (131072 / (8 * TILEB));
  using Cfg = MmaCfg<D, KVT, NN, 4, NS>;
  KernelInfo k = info_of<Cfg>(&decode_mma_kernel<D, KVT, NN, 4, NS>, true);
  k.box_cols = Cfg::BOXCOLS;
  k.swizzle = Cfg::BOXB == 128 ? 128 : 64;
  return k;
}

template <int D, int KVT>
KernelInfo pick(int impl, int g) {
  if (impl == PA_DECODE_SIMT) {
    if (g <= 1) return simt_info<D, KVT, 1>();
    if (g <= 2) return simt_info<D, KVT, 2>();
    return simt_info<D, KVT, 4>();
  }
  if (g <= 8) return mma_info<D, KVT, 1>();
  return mma_info<D, KVT, 2>();
}

KernelInfo kernel_for(const pa_kv_desc &d, int impl) {
  const int g = d.num_q_heads / d.num_kv_heads;
  const bool bf = d.kv_dtype == PA_KV_BF16;
  if (d.head_dim == 128) return bf ? pick<128, kKvBf16>(impl, g) : pick<128, kKvFp8>(impl, g);
  return bf ? pick<64, kKvBf16>(impl, g) : pick<64, kKvFp8>(impl, g);
}

int resolve_impl(const pa_kv_desc &d) {
  if (d.decode_impl != PA_DECODE_AUTO) return d.decode_impl;
  return PA_DECODE_MMA;
}

// cuTensorMapEncodeTiled, fetched from the driver through the runtime
using EncodeTiledFn = CUresult (*)(CUtensorMap *, CUtensorMapDataType, cuuint32_t, void *, const cuuint64_t *,
                                   const cuuint64_t *, const cuuint32_t *, const cuuint32_t *, CUtensorMapInterleave,
                                   CUtensorMapSwizzle, CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

EncodeTiledFn encode_tiled() {
  static EncodeTiledFn fn = [] {
    void *p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) != cudaSuccess ||
        q != cudaDriverEntryPointSuccess)
      p = nullptr;
    return reinterpret_cast<EncodeTiledFn>(p);
  }();
  return fn;
}

bool make_cache_map(CUtensorMap *map, const void *base, const pa_kv_desc &d, const KernelInfo &k) {
  EncodeTiledFn enc = encode_tiled();
  if (!enc) return false;
  const bool bf = d.kv_dtype == PA_KV_BF16;
  const int esz = bf ? 2 : 1;
  const cuuint64_t rows = static_cast<cuuint64_t>(d.num_blocks) * d.num_kv_heads * 16;
  const cuuint64_t dims[2] = {static_cast<cuuint64_t>(d.head_dim), rows};
  const cuuint64_t strides[1] = {static_cast<cuuint64_t>(d.head_dim) * esz};
  const cuuint32_t box[2] = {static_cast<cuuint32_t>(k.box_cols), 16};
  const cuuint32_t estr[2] = {1, 1};
  const CUresult r = enc(map, bf ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16 : CU_TENSOR_MAP_DATA_TYPE_UINT8, 2,
                         const_cast<void *>(base), dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
                         k.swizzle == 128 ? CU_TENSOR_MAP_SWIZZLE_128B : CU_TENSOR_MAP_SWIZZLE_64B,
                         CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS;
}

}  // namespace

int device_sm_count() { return device_info().sm_count; }

pa_status plan_decode(const pa_kv_desc &d, int32_t num_seqs, DecodePlan *plan, const char **why) {
  const int g = d.num_q_heads / d.num_kv_heads;
  const int impl = resolve_impl(d);
  if (impl != PA_DECODE_SIMT && impl != PA_DECODE_MMA) {
    *why = "decode_impl must be PA_DECODE_AUTO, PA_DECODE_SIMT or PA_DECODE_MMA";
    return PA_ERR_INVALID_ARG;
  }
  if (impl == PA_DECODE_SIMT && g > 4) {
    *why = "the CUDA-core decode kernel supports group sizes up to 4";
    return PA_ERR_UNSUPPORTED;
  }
  if (impl == PA_DECODE_MMA && static_cast<int64_t>(d.num_blocks) * d.num_kv_heads * 16 > 0x7fffffffLL) {
    *why = "the tensor-core decode kernel addresses at most 2^31 cache rows";
    return PA_ERR_UNSUPPORTED;
  }
  const KernelInfo k = kernel_for(d, impl);
  if (cudaFuncSetAttribute(k.fn, cudaFuncAttributeMaxDynamicSharedMemorySize, static_cast<int>(k.smem)) != cudaSuccess) {
    *why = "cudaFuncSetAttribute(MaxDynamicSharedMemorySize) failed";
    return PA_ERR_CUDA;
  }
  int occ = 0;
  if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&occ, k.fn, k.threads, k.smem) != cudaSuccess || occ < 1) {
    *why = "the decode kernel does not fit on this device";
    return PA_ERR_CUDA;
  }
  plan->impl = impl;
  plan->group_pad = k.hp;
  plan->num_ctas = device_info().sm_count * occ;
  plan->workspace_bytes = ws_layout(num_seqs, d.num_kv_heads, plan->num_ctas, k.hp, d.head_dim).total;
  return PA_OK;
}

cudaError_t launch_decode(const pa_kv_desc &d, const DecodePlan &plan, float *out, float *lse,
                          const void *q, const void *k_cache, const void *v_cache,
                          const int32_t *block_tables, int32_t max_blocks_per_seq,
                          const int32_t *context_lens, int32_t num_seqs, float scale,
                          void *workspace, cudaStream_t stream) {
  const KernelInfo k = kernel_for(d, plan.impl);
  const WsLayout w = ws_layout(num_seqs, d.num_kv_heads, plan.num_ctas, plan.group_pad, d.head_dim);
  uint8_t *ws = static_cast<uint8_t *>(workspace);
  DecodeArgs a;
  memset(&a, 0, sizeof a);
  if (k.mma) {
    if (!make_cache_map(&a.kmap, k_cache, d, k) || !make_cache_map(&a.vmap, v_cache, d, k))
      return cudaErrorInvalidValue;
  }
  a.out = out;
  a.lse = lse;
  a.q = static_cast<const uint16_t *>(q);
  a.k_cache = static_cast<const uint8_t *>(k_cache);
  a.v_cache = static_cast<const uint8_t *>(v_cache);
  a.block_tables = block_tables;
  a.context_lens = context_lens;
  a.max_blocks_per_seq = max_blocks_per_seq;
  a.num_seqs = num_seqs;
  a.num_kv_heads = d.num_kv_heads;
  a.num_q_heads = d.num_q_heads;
  a.g = d.num_q_heads / d.num_kv_heads;
  const bool fp8 = d.kv_dtype == PA_KV_FP8_E4M3;
  const float ks = (fp8 && d.k_scale != 0.f) ? d.k_scale : 1.f;
  a.qscale = scale * ks * kLog2e;
  a.vscale = (fp8 && d.v_scale != 0.f) ? d.v_scale : 1.f;
  a.err = reinterpret_cast<int32_t *>(ws);
  a.seg_counter = reinterpret_cast<int32_t *>(ws + w.counter_off);
  a.slot_lse = reinterpret_cast<float *>(ws + w.slot_lse_off);
  a.slot_o = reinterpret_cast<float *>(ws + w.slot_o_off);
  void *args[] = {&a};
  return cudaLaunchKernel(k.fn, dim3(plan.num_ctas), dim3(k.threads), args, k.smem, stream);
}

}  // namespace pa
