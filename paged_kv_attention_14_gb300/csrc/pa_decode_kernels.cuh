// pa_decode_kernels.cuh -- split-KV decode attention over the block-paged KV cache.
//
// What it computes: for every sequence s and query head h,
//   out[s][h] = sum_t softmax_t(scale * q[s][h] . K_t) V_t
// over the tokens t < context_lens[s] of kv head h / g, gathered through the
// sequence's block table.  This is the "paged attention (block-paged KV
// cache)" of the vllm.cpp implementation notes ("What's implemented", Model
// forward bullet) over its "Block-Paged KV Cache (FP8/FP16)" (architecture
// figure of "Building and Deploying vllm.cpp ..."), block size 16.  With FP8
// pages ("fp8 halves page size to 1 byte per element", CLI table of the same
// walkthrough) the E4M3 / E5M2 bytes are decoded inside the load and the
// scales (per tensor, or per kv head) are folded into the softmax scale (K)
// and the output (V).  fp16 pages (an fp16 model) take fp16 MMAs.  Local
// attention (sliding window, chunked-local) starts each sequence's stream at
// the block of its first visible key.
//
// How (GB300 design, not taken from the pages):
//  * Persistent grid, stream-K work split.  A segment is (sequence, group of
//    HG kv heads); the (segment, block) list is flattened in sequence-major
//    order and cut into gridDim.x equal contiguous ranges; each CTA owns one
//    range, so a 131072-token sequence next to short ones is balanced to
//    within one block.  A range cuts a segment into at most two pieces per
//    CTA; pieces are written to per-CTA slots and the last CTA to finish a
//    segment (an atomic counter, no waiting) merges them by log-sum-exp in
//    the same launch.  Each CTA streams the piece at the end of its range
//    first, so that most merges overlap the stream.
//  * One producer warp streams KV with the TMA engine into an NS-stage
//    shared-memory ring guarded by mbarriers.  In this cache layout the HG kv
//    heads of one block are contiguous, so one copy moves a block for a whole
//    head group (16 KB for 4 bf16 heads of 128); the block table is read 32
//    entries at a time, the next 32 requested while the current ones are
//    used, and the producer runs ahead across piece boundaries.
//  * Two consumers share that framework:
//    - SIMT (group size <= 4, HG = 1): fp32 CUDA-core dot products; 8 lanes
//      share a token row, three xor-shuffles reduce it.
//    - MMA (group size <= 16): each consumer warp owns one kv head of the
//      group and one 16-token block per stage: S^T = K Q^T and O^T += V^T P^T
//      as m16n8k16 tensor-core MMAs with the tokens as M and the query heads
//      of the group as N (padded to 8 or 16); P^T comes from the S^T
//      accumulators by an in-register 8x8 transpose (movmatrix).  Tiles
//      arrive 128B/64B-swizzled, so every ldmatrix is bank-conflict free.
//      bf16 / fp16 KV uses MMAs of that type with the probabilities split into
//      a hi + lo pair (near-fp32 accuracy); 8-bit KV is converted exactly to
//      f16 in registers and uses f16 MMAs.  A separate epilogue warp folds the
//      consumer warps' partial states of each finished piece and writes the
//      output or the slot (and merges), so consumers never stop streaming.
#pragma once

#include <cuda.h>
#include <float.h>
#include <string.h>

#include "pa_device.cuh"
#include "pa_internal.h"

namespace pa {
namespace dec {

constexpr float kLog2e = 1.4426950408889634f;
constexpr float kLn2 = 0.6931471805599453f;
constexpr int kFlagFirst = 1;
constexpr int kFlagLast = 2;
constexpr int kFlagEnd = 4;  // the stage holds the sequence's last token
constexpr int kStageData = 0;
constexpr int kStageEnd = 1;
constexpr int kConsumerWarps = 4;

struct __align__(16) StageHdr {
  long long seg_start;  // flat block index where the segment starts
  int kind;
  int s;
  int grp;     // kv head group (kv heads grp * HG .. grp * HG + HG - 1)
  int ntok;    // tokens of this stage before the sequence's end
  int flags;   // kFlagFirst / kFlagLast of a piece, kFlagEnd
  int seg_nb;  // blocks of the segment
  int tlo;     // tokens at the stage's start before the first key (local attention)
};

struct DecodeArgs {
  CUtensorMap kmap;  // MMA kernel only: the K cache (see make_cache_map)
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
  int g;           // query heads per kv head
  int num_groups;  // kv head groups per sequence (num_kv_heads / HG)
  float qscale;    // scale * k_scale * log2(e)
  float vscale;    // v_scale (1 for bf16)
  float qscale0;   // scale * log2(e): qscale before the k scale
  const float *k_scales;  // per-kv-head scales of an 8-bit cache (NULL: k_scale, v_scale)
  const float *v_scales;
  int window;      // sliding window (0: none)
  int chunk;       // chunked-local attention (0: none)
  int32_t *err;          // the workspace's error word
  int32_t *user_err;     // the caller's error word (pa_kv_desc.error_word), or NULL
  unsigned long long wait_ns;  // limit of every bounded wait
  int checked;     // range-check block ids and lengths (pa_kv_desc.check_indices)
  int stall;       // test hook: the producer issues nothing, so the waits run out
  int num_blocks;  // blocks of the cache (checked mode)
  int32_t *seg_counter;  // [num_seqs * num_groups] pieces of each split segment finished
  float *slot_lse;       // [grid][2][slot heads], log2 domain
  float *slot_o;         // [grid][2][slot heads][D]
  // pa_decode_append (MMA kernel): sequence s's token at position
  // context_lens[s] - 1 is k_new[s] / v_new[s] ([S][kv heads][D], the
  // activation type); the consumer of the sequence's last block puts it into
  // its staged tile and into the cache (k_write / v_write, the caches), an
  // 8-bit cache's row encoded as pa_cache_write encodes it, with the
  // per-tensor scales k_enc / v_enc or the per-head k_scales / v_scales.
  // NULL: nothing to append.
  const uint8_t *k_new;
  const uint8_t *v_new;
  uint8_t *k_write;
  uint8_t *v_write;
  float k_enc;
  float v_enc;
};

// Optional timeline counters (compiled only with -DPA_DECODE_TRACE): per CTA,
// [0] consumer warp 0 cycles waiting for a full stage, [1] its cycles handing
// pieces over, [2] its total cycles, [3] producer cycles waiting for an
// empty stage, [4] producer cycles waiting for block-table loads, [5]
// producer total cycles, [6] stages consumed, [7] pieces finished.
#ifdef PA_DECODE_TRACE
static __device__ unsigned long long g_pa_trace[4096][8];
#define PA_TRACE(...) __VA_ARGS__
#else
#define PA_TRACE(...)
#endif

// Blocks of a sequence of L tokens the decode query reads: from the block
// holding its first key (local attention) to the last one.
__device__ __forceinline__ int seq_first_block(const DecodeArgs &a, int L) {
  return local_first_key(L - 1, a.window, a.chunk) >> 4;
}
__device__ __forceinline__ int seq_blocks(const DecodeArgs &a, int L) {
  return ((L + 15) >> 4) - seq_first_block(a, L);
}

// Score and output scales of kv head kvh: its per-head k / v scale where the
// cache has them, else the per-tensor ones folded in on the host.
__device__ __forceinline__ float head_qscale(const DecodeArgs &a, int kvh) {
  return a.k_scales ? a.qscale0 * __ldg(a.k_scales + kvh) : a.qscale;
}
__device__ __forceinline__ float head_vscale(const DecodeArgs &a, int kvh) {
  return a.v_scales ? __ldg(a.v_scales + kvh) : a.vscale;
}

// Error bits into the workspace's error word and the caller's.
__device__ __forceinline__ void report(const DecodeArgs &a, int bits) { report_error(a.err, a.user_err, bits); }

// Context length of sequence s; in checked mode clamped to the block table's
// capacity (and reported when outside it).
__device__ __forceinline__ int seq_len(const DecodeArgs &a, int s) {
  const int L = __ldg(a.context_lens + s);
  return a.checked ? checked_len(L, a.max_blocks_per_seq * 16, a.err, a.user_err) : L;
}

// ---------------------------------------------------------------- workspace

constexpr size_t align256(size_t x) { return (x + 255) & ~size_t(255); }

// Workspace: [0, 4) error word, then the merge counters (one per segment;
// every merge resets its counter, so they stay zero between launches), slot
// lse and slot outputs.
struct WsLayout {
  size_t counter_off, slot_lse_off, slot_o_off, total;
};

// slot_heads: query heads of one slot (kv heads per group x padded group size)
inline WsLayout ws_layout(int num_seqs, int num_groups, int grid, int slot_heads, int d) {
  WsLayout w;
  w.counter_off = 256;
  w.slot_lse_off = w.counter_off + align256(sizeof(int32_t) * size_t(num_seqs) * num_groups);
  w.slot_o_off = w.slot_lse_off + align256(sizeof(float) * size_t(grid) * 2 * slot_heads);
  w.total = w.slot_o_off + align256(sizeof(float) * size_t(grid) * 2 * slot_heads * d);
  return w;
}

// Output of an empty sequence: zeros and lse = -inf.
__device__ inline void zero_sequence(const DecodeArgs &a, int s, int D) {
  for (int h = 0; h < a.num_q_heads; ++h) {
    float *o = a.out + (static_cast<int64_t>(s) * a.num_q_heads + h) * D;
    for (int d = 0; d < D; ++d) o[d] = 0.f;
    if (a.lse) a.lse[static_cast<int64_t>(s) * a.num_q_heads + h] = -INFINITY;
  }
}

// --------------------------------------------------------- shared framework

// Pass over context_lens by one warp: the number of 16-token blocks of all
// sequences; empty sequences are zero-filled by the CTA (or partition) me
// = s % G of the G that split the work.
template <int D>
__device__ long long count_blocks(const DecodeArgs &a, int lane, int me, int G) {
  long long nb_sum = 0;
  const int S = a.num_seqs;
  for (int base = 0; base < S; base += 256) {
    unsigned acc = 0;
#pragma unroll
    for (int i = 0; i < 8; ++i) {
      const int s = base + i * 32 + lane;
      if (s < S) {
        const int L = seq_len(a, s);
        if (L > 0)
          acc += static_cast<unsigned>(seq_blocks(a, L));
        else if (s % G == me)
          zero_sequence(a, s, D);
      }
    }
    nb_sum += __reduce_add_sync(0xffffffffu, acc);
  }
  return nb_sum;
}

// The producer warp: walks this CTA's range of flat (sequence, head group,
// block) units and fills the stage ring.  Cfg::issue() starts the copies of
// one block's K and V for the head group (one lane per block).
//
// Order: when the range ends inside a segment that starts inside it (a
// segment split with the next CTA), that piece is streamed first and the
// rest of the range after it.  The next CTA streams its own piece of such a
// segment early as well, so the segment's merge (done by whichever CTA
// finishes the segment's last piece) overlaps the stream instead of trailing
// the launch.
template <class Cfg>
__device__ void produce(const DecodeArgs &a, uint8_t *stages, StageHdr *hdr, uint64_t *full,
                        uint64_t *empty, long long per_cta, long long total, int lane, int me) {
  constexpr int NS = Cfg::NS;
  constexpr int BPS = Cfg::BPS;
  const int S = a.num_seqs;
  const int NG = a.num_groups;
  const long long b0 = static_cast<long long>(me) * per_cta;
  const long long b1 = min(b0 + per_cta, total);
  const uint64_t pol = l2_evict_first_policy();
  // test hook: issue nothing and signal nothing, so that every consumer
  // wait runs out (nothing is in flight when the kernel gives up)
  if (a.stall) return;
  int stage = 0;
  uint32_t ppar = 1;  // a fresh barrier counts its preceding phase (parity 1) as complete
  bool ok = true;
  int issued = 0;
  PA_TRACE(const long long tp0 = clock64(); long long tp_empty = 0, tp_table = 0;)
  if (b0 < b1) {
    // one pass over the sequences: the sequences holding flat units b0 and
    // b1 - 1, and the flat start of each
    long long pre0 = 0, prez = 0;
    int s0 = -1, sz = -1;
    {
      long long pre = 0;
      for (int base = 0; base < S && sz < 0; base += 32) {
        const int si = base + lane;
        const int Li = si < S ? seq_len(a, si) : 0;
        const long long v = Li > 0 ? static_cast<long long>(seq_blocks(a, Li)) * NG : 0;
        long long incl = v;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
          const long long t = __shfl_up_sync(0xffffffffu, incl, o);
          if (lane >= o) incl += t;
        }
        const long long excl = incl - v;
        const unsigned m0 = __ballot_sync(0xffffffffu, v > 0 && pre + excl <= b0 && b0 < pre + incl);
        const unsigned mz = __ballot_sync(0xffffffffu, v > 0 && pre + excl <= b1 - 1 && b1 - 1 < pre + incl);
        if (s0 < 0 && m0) {
          const int src = __ffs(m0) - 1;
          s0 = base + src;
          pre0 = pre + __shfl_sync(0xffffffffu, excl, src);
        }
        if (mz) {
          const int src = __ffs(mz) - 1;
          sz = base + src;
          prez = pre + __shfl_sync(0xffffffffu, excl, src);
        }
        pre += __shfl_sync(0xffffffffu, incl, 31);
      }
    }
    // walking state: sequence s (flat start pre, L tokens, blocks [fb, fb + nb)),
    // head group grp, block offset off within the segment
    int s = 0, L = 0, fb = 0, nb = 1, grp = 0, off = 0;
    long long pre = 0;
    auto locate = [&](int s_, long long pre_, long long pos) {
      s = s_;
      pre = pre_;
      L = seq_len(a, s);
      fb = seq_first_block(a, L);
      nb = ((L + 15) >> 4) - fb;
      grp = static_cast<int>((pos - pre) / nb);
      off = static_cast<int>((pos - pre) % nb);
    };
    // block-table window: entries [wb, wb + 32) in w_cur and [wb + 32, wb + 64)
    // in w_nxt, one per lane; the next 32 are requested while the current
    // ones are used.  (Reading w_nxt every stage stalls the producer briefly
    // after each window move; a variant that avoided those stalls and kept
    // each sequence's first window for its later head groups streamed 2-5%
    // slower on GB300, the producer running further ahead of the consumers.)
    int win_s = -1, wb = 0, w_cur = 0, w_nxt = 0;
    const int32_t *trow = a.block_tables;
    auto tload = [&](int e) {
      if (e >= fb + nb) return 0;
      const int v = __ldg(trow + e);
      return a.checked ? checked_block(v, a.num_blocks, a.err, a.user_err) : v;
    };
    // streams flat units [from, to), starting from the located state
    auto stream = [&](long long from, long long to) {
      long long cur = from;
      while (cur < to && ok) {
        const long long seg_start = pre + static_cast<long long>(grp) * nb;
        const long long piece_end = min(to, seg_start + nb);
        const int npb = static_cast<int>(piece_end - cur);
        for (int k = 0; k < npb; k += BPS) {
          const int nblk = min(BPS, npb - k);
          const int lb0 = fb + off + k;  // logical block of the stage's first block
          PA_TRACE(const long long tt0 = clock64();)
          if (win_s != s || lb0 < wb || lb0 + nblk > wb + 64) {
            trow = a.block_tables + static_cast<int64_t>(s) * a.max_blocks_per_seq;
            win_s = s;
            wb = lb0;
            w_cur = tload(wb + lane);
            w_nxt = tload(wb + 32 + lane);
          }
          const int rel = lb0 - wb + lane;  // this lane's block, relative to the window
          const int v_cur = __shfl_sync(0xffffffffu, w_cur, rel & 31);
          const int v_nxt = __shfl_sync(0xffffffffu, w_nxt, rel & 31);
          const int phys = rel < 32 ? v_cur : v_nxt;
          if (lb0 + nblk >= wb + 32) {  // the next stage starts in the second half
            wb += 32;
            w_cur = w_nxt;
            w_nxt = tload(wb + 32 + lane);
          }
          PA_TRACE(const long long tt1 = clock64(); tp_table += tt1 - tt0;)
          if (!mbar_wait(&empty[stage], ppar, a.wait_ns)) {
            ok = false;
            break;
          }
          PA_TRACE(tp_empty += clock64() - tt1;)
          const bool first = (k == 0);
          const uint32_t qbytes = static_cast<uint32_t>(Cfg::HG * a.g * Cfg::D * 2);
          if (lane == 0) {
            StageHdr h;
            h.seg_start = seg_start;
            h.kind = kStageData;
            h.s = s;
            h.grp = grp;
            h.ntok = min(L - lb0 * 16, nblk * 16);
            h.flags = (first ? kFlagFirst : 0) | (k + BPS >= npb ? kFlagLast : 0) |
                      (L - lb0 * 16 <= nblk * 16 ? kFlagEnd : 0);
            h.seg_nb = nb;
            h.tlo = max(0, local_first_key(L - 1, a.window, a.chunk) - lb0 * 16);
            hdr[stage] = h;
            mbar_arrive_expect_tx(&full[stage], 2u * nblk * Cfg::GTILE + (first ? qbytes : 0u));
          }
          __syncwarp();
          uint8_t *sk = stages + size_t(stage) * Cfg::STAGEB;
          if (lane < nblk) Cfg::issue(a, sk, lane, phys, grp, &full[stage], pol);
          if (first && lane == 31) {
            const uint16_t *qsrc = a.q + (static_cast<int64_t>(s) * a.num_q_heads + grp * Cfg::HG * a.g) * Cfg::D;
            bulk_g2s(sk + Cfg::QOFF, qsrc, qbytes, &full[stage]);
          }
          ++issued;
          if (++stage == NS) {
            stage = 0;
            ppar ^= 1;
          }
        }
        cur = piece_end;
        off = 0;
        if (++grp == NG) {
          grp = 0;
          pre += static_cast<long long>(nb) * NG;
          do {
            ++s;
          } while (s < S && seq_len(a, s) <= 0);
          if (s < S) {
            L = seq_len(a, s);
            fb = seq_first_block(a, L);
            nb = ((L + 15) >> 4) - fb;
          }
        }
      }
    };
    // the segment holding the range's last unit
    const int nbz = seq_blocks(a, seq_len(a, sz));
    const long long segz = prez + (b1 - 1 - prez) / nbz * nbz;
    if (segz > b0 && segz + nbz > b1) {
      locate(sz, prez, segz);
      stream(segz, b1);
      locate(s0, pre0, b0);
      stream(b0, segz);
    } else {
      locate(s0, pre0, b0);
      stream(b0, b1);
    }
  }
  if (ok) {
    if (mbar_wait(&empty[stage], ppar, a.wait_ns)) {
      if (lane == 0) {
        hdr[stage].kind = kStageEnd;
        mbar_arrive(&full[stage]);
      }
    } else {
      ok = false;
    }
  }
  PA_TRACE(if (lane == 0) {
    g_pa_trace[me][3] = tp_empty;
    g_pa_trace[me][4] = tp_table;
    g_pa_trace[me][5] = clock64() - tp0;
  })
  if (!ok) {
    if (lane == 0) report(a, kErrWaitTimeout);
    // let the copies already issued land before the CTA can exit
    for (int i = 1; i <= min(issued, NS); ++i) {
      int st = stage - i;
      uint32_t par = ppar ^ 1;
      if (st < 0) {
        st += NS;
        par ^= 1;
      }
      mbar_wait(&full[st], par, a.wait_ns);
    }
  }
}

// Finish one piece on the SIMT consumer warps.  NP partial states lie in
// red[0..NP) (one per warp): for every head j of the group, unnormalised
// O[j][0..D), the running max m (log2 domain) at [D] and the sum l at [D+1]
// (head stride D + 2, HP heads per partial).  Combines them, then writes the
// output (whole segment in this CTA) or this CTA's slot, and the last CTA of
// a split segment merges all slots of that segment.
template <int D, int HP, int NP, int NC>
__device__ void finish_piece(const DecodeArgs &a, const StageHdr &h, const float *red, long long per_cta,
                             int *s_flag, int tid, int me) {
  constexpr int CT = NC * 32;
  constexpr int REDW = HP * (D + 2);
  const long long c1 = h.seg_start / per_cta;
  const long long c2 = (h.seg_start + h.seg_nb - 1) / per_cta;
  const bool split = c1 != c2;
  const int my_slot = (h.seg_start <= static_cast<long long>(me) * per_cta) ? 0 : 1;
  const int hq0 = h.grp * a.g;
  for (int idx = tid; idx < a.g * D; idx += CT) {
    const int j = idx / D;
    const int d = idx - j * D;
    float M = -INFINITY;
#pragma unroll
    for (int w = 0; w < NP; ++w) M = fmaxf(M, red[w * REDW + j * (D + 2) + D]);
    float Ls = 0.f, O = 0.f;
#pragma unroll
    for (int w = 0; w < NP; ++w) {
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
      a.out[(static_cast<int64_t>(h.s) * a.num_q_heads + hq0 + j) * D + d] = res * head_vscale(a, h.grp);
      if (a.lse && d == 0) a.lse[static_cast<int64_t>(h.s) * a.num_q_heads + hq0 + j] = lse2 * kLn2;
    } else {
      const int64_t sl = (static_cast<int64_t>(me) * 2 + my_slot) * HP + j;
      a.slot_o[sl * D + d] = res;
      if (d == 0) a.slot_lse[sl] = lse2;
    }
  }
  if (split) {
    named_bar_sync(1, CT);
    if (tid == 0) {
      const int seg = h.s * a.num_groups + h.grp;
      const int npieces = static_cast<int>(c2 - c1 + 1);
      const int prev = atom_add_acq_rel_gpu(a.seg_counter + seg, 1);
      const int last = prev == npieces - 1;
      if (last) st_relaxed_gpu(a.seg_counter + seg, 0);  // ready for the next launch
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
        a.out[(static_cast<int64_t>(h.s) * a.num_q_heads + hq0 + j) * D + d] = O / W * head_vscale(a, h.grp);
        if (a.lse && d == 0) a.lse[static_cast<int64_t>(h.s) * a.num_q_heads + hq0 + j] = (M + log2f(W)) * kLn2;
      }
    }
  }
  named_bar_sync(1, CT);  // the reduction buffer is free again
}

// Kernel prologue shared by both consumers: barrier init, block count,
// per-CTA range (G CTAs or partitions split the work; this is number me).
// Returns per_cta and (for the producer warp) the total.
template <class Cfg>
__device__ long long prologue(const DecodeArgs &a, uint64_t *full, uint64_t *empty, long long *total_out,
                              long long *s_per_cta, int me, int G) {
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
    const long long nb_sum = count_blocks<Cfg::D>(a, tid & 31, me, G);
    *total_out = nb_sum * a.num_groups;
    if ((tid & 31) == 0) *s_per_cta = (*total_out + G - 1) / G;
  }
  __syncthreads();
  return *s_per_cta;
}

// ============================================================ SIMT consumer

// Which head_dim elements lane j8 (0..7) of an 8-lane token group holds, and
// how it loads them from a cached row.  2-byte rows (bf16, fp16): 16-byte
// chunks j8, j8 + 8, ... (each quarter-warp reads one contiguous 128-byte
// span).  8-bit rows: one contiguous run of D/8 bytes per lane.
template <int D, int KVT>
struct RowSlice {
  static constexpr int EPL = D / 8;
  __device__ static __forceinline__ int dim(int j8, int e) {
    if (kv16(KVT)) return ((e >> 3) * 8 + j8) * 8 + (e & 7);
    return j8 * EPL + e;
  }
  __device__ static __forceinline__ void load(const uint8_t *row, int j8, float (&x)[EPL]) {
    if constexpr (kv16(KVT)) {
#pragma unroll
      for (int c = 0; c < EPL / 8; ++c) {
        const uint4 u = *reinterpret_cast<const uint4 *>(row + (c * 8 + j8) * 16);
        x[c * 8 + 0] = lo16<KVT>(u.x);
        x[c * 8 + 1] = hi16<KVT>(u.x);
        x[c * 8 + 2] = lo16<KVT>(u.y);
        x[c * 8 + 3] = hi16<KVT>(u.y);
        x[c * 8 + 4] = lo16<KVT>(u.z);
        x[c * 8 + 5] = hi16<KVT>(u.z);
        x[c * 8 + 6] = lo16<KVT>(u.w);
        x[c * 8 + 7] = hi16<KVT>(u.w);
      }
    } else if (EPL == 16) {
      const uint4 u = *reinterpret_cast<const uint4 *>(row + j8 * 16);
      const uint32_t w[4] = {u.x, u.y, u.z, u.w};
#pragma unroll
      for (int c = 0; c < 4; ++c) {
        fp8x2_to_f32<KVT>(static_cast<uint16_t>(w[c] & 0xffffu), x[4 * c + 0], x[4 * c + 1]);
        fp8x2_to_f32<KVT>(static_cast<uint16_t>(w[c] >> 16), x[4 * c + 2], x[4 * c + 3]);
      }
    } else {
      const uint2 u = *reinterpret_cast<const uint2 *>(row + j8 * 8);
      const uint32_t w[2] = {u.x, u.y};
#pragma unroll
      for (int c = 0; c < 2; ++c) {
        fp8x2_to_f32<KVT>(static_cast<uint16_t>(w[c] & 0xffffu), x[4 * c + 0], x[4 * c + 1]);
        fp8x2_to_f32<KVT>(static_cast<uint16_t>(w[c] >> 16), x[4 * c + 2], x[4 * c + 3]);
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
  static constexpr int ESZ = kv16(KVT) ? 2 : 1;
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
  static constexpr int HG = 1;   // kv heads per stage group
  static constexpr int GTILE = TILEB;
  static constexpr int SLOTH = GP_;
  static_assert(TPG >= 1 && TPG * NG == BPS * 16, "stage must split evenly over groups");
  static_assert(BPS <= 31, "one producer lane per block plus one for q");

  static constexpr int GQ = GP_;  // query heads of a group the q area holds
  __device__ static __forceinline__ void issue(const DecodeArgs &a, uint8_t *sk, int i, int phys, int grp,
                                               uint64_t *bar, uint64_t pol) {
    const int64_t tile = (static_cast<int64_t>(phys) * a.num_kv_heads + grp) * TILEB;
    bulk_g2s(sk + i * TILEB, a.k_cache + tile, TILEB, bar, pol);
    bulk_g2s(sk + KVB + i * TILEB, a.v_cache + tile, TILEB, bar, pol);
  }
};

template <int D, int KVT, int GP, int BPS, int NS>
__global__ void __launch_bounds__((kConsumerWarps + 1) * 32, 2) decode_simt_kernel(const __grid_constant__ DecodeArgs a) {
  using C = SimtCfg<D, KVT, GP, BPS, NS>;
  using RS = RowSlice<D, KVT>;
  // launched as a programmatic dependent of the preceding kernel in the
  // stream: nothing is read before that kernel's writes are visible
  asm volatile("griddepcontrol.wait;" ::: "memory");
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
  const int me = blockIdx.x;
  const long long per_cta = prologue<C>(a, full, empty, &total, &s_per_cta, me, gridDim.x);
  if (warp == NC) {
    produce<C>(a, stages, hdr, full, empty, per_cta, total, lane, me);
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
    if (!mbar_wait(&full[stage], cpar, a.wait_ns)) {
      if (lane == 0) report(a, kErrWaitTimeout);
      break;
    }
    const StageHdr h = hdr[stage];
    if (h.kind == kStageEnd) break;
    const uint8_t *Ks = stages + size_t(stage) * C::STAGEB;
    const uint8_t *Vs = Ks + C::KVB;
    if (h.flags & kFlagFirst) {
      const uint16_t *Qs = reinterpret_cast<const uint16_t *>(Ks + C::QOFF);
      const float qsc = head_qscale(a, h.grp);  // one kv head per segment
#pragma unroll
      for (int j = 0; j < GP; ++j) {
        m[j] = -INFINITY;
        l[j] = 0.f;
#pragma unroll
        for (int e = 0; e < EPL; ++e) {
          q[j][e] = j < a.g ? lo16<KVT == kKvF16 ? kKvF16 : kKvBf16>(Qs[j * D + RS::dim(j8, e)]) * qsc : 0.f;
          o[j][e] = 0.f;
        }
      }
    }
    float x[C::TPG][GP];
#pragma unroll
    for (int i = 0; i < C::TPG; ++i) {
      const int r = gid + C::NG * i;
      const bool valid = r < h.ntok && r >= h.tlo;
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
      if (r < h.ntok && r >= h.tlo) {
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
    finish_piece<D, C::HP, NC, NC>(a, h, red, per_cta, &s_flag, tid, me);
  }
}

// ============================================================= MMA consumer

// How a head-group tile of 256-byte rows (bf16, head_dim 128) is copied:
//   kWideHalfMajor  one 3-D box {64 columns, HG*16 rows, 2 halves} (row
//                   stride 256 B, half stride 128 B); lands as
//                   [half][row][128 B], bank-conflict free
//   kWideTokMajor   one 3-D box {64 columns, 2 halves, HG*16 rows} (strides
//                   128 B, 256 B); lands as [row][half][128 B]; ldmatrix
//                   reads see 2-way bank conflicts
//   kWideTwoBoxes   two 2-D boxes {64 columns, HG*16 rows}, one per half;
//                   lands as [half][row][128 B]
constexpr int kWideHalfMajor = 0;
constexpr int kWideTokMajor = 1;
constexpr int kWideTwoBoxes = 2;
constexpr int kWideMode = kWideHalfMajor;

// Byte offset of 16-byte chunk `ch` of row `row` (row = head of the group *
// 16 + token) of a head-group tile as TMA lays it down with 128-byte swizzle
// (within every 1024 bytes the 16-byte chunk index is XORed with the 128-byte
// row index) or 64-byte swizzle (chunk XOR bits 7-8 of the address).
template <int ROWB, int HG>
__device__ __forceinline__ uint32_t swz_off(int row, int ch) {
  if constexpr (ROWB > 128 && kWideMode == kWideTokMajor) {
    const int rr = 2 * row + (ch >> 3);
    return static_cast<uint32_t>(rr * 128 + (((ch & 7) ^ (rr & 7)) << 4));
  } else if constexpr (ROWB > 128) {
    return static_cast<uint32_t>((ch >> 3) * (HG * 16 * 128) + row * 128 + (((ch & 7) ^ (row & 7)) << 4));
  } else if constexpr (ROWB == 128) {
    return static_cast<uint32_t>(row * 128 + ((ch ^ (row & 7)) << 4));
  } else {
    return static_cast<uint32_t>(row * 64 + ((ch ^ ((row >> 1) & 3)) << 4));
  }
}

// D: head_dim; KVT: cache type; GQ: largest group size served (4, 8 or 16,
// rounded up to the MMA's 8-wide n-tiles); HG: kv heads per stage; NS: stages.
template <int D_, int KVT_, int GQ_, int HG_, int NS_, int NC_>
struct MmaCfg {
  static constexpr int D = D_;
  static constexpr int KVT = KVT_;
  static constexpr int GQ = GQ_;           // query heads per kv head held in smem
  static constexpr int NN = (GQ_ + 7) / 8;  // n-tiles of 8 query heads in the MMAs
  static constexpr int HG = HG_;
  static constexpr int NS = NS_;
  static constexpr int NC = NC_;  // consumer warps; warp NC produces, NC + 1 finishes
  static constexpr int BPS = NC / HG;        // blocks per stage: one (block, head) tile per consumer warp
  static constexpr int ESZ = kv16(KVT) ? 2 : 1;
  static constexpr int ROWB = D * ESZ;
  static constexpr int TILEB = 16 * ROWB;    // one (block, kv head)
  static constexpr int GTILE = HG * TILEB;   // one block of a head group: one copy
  static constexpr int KVB = BPS * GTILE;
  static constexpr int QB = ((HG * GQ * D * 2 + 1023) / 1024) * 1024;
  static constexpr int QOFF = 2 * KVB;
  static constexpr int STAGEB = 2 * KVB + QB;
  static constexpr int NTHREADS = (NC + 2) * 32;
  static constexpr int RSTR = D + 4;         // floats per head row of a partial: O[D], m, l, pad
  static constexpr int REDW = GQ * RSTR;     // floats of one warp's partial
  static constexpr int SLOTH = HG * GQ;      // query heads of a slot
  static constexpr size_t SMEM = 1024 + size_t(NS) * STAGEB + size_t(2) * NC * REDW * sizeof(float) +
                                 (NS + 2) * sizeof(StageHdr) + 2 * (NS + 2) * sizeof(uint64_t) + 16;
  static_assert(NC % HG == 0, "consumer warps split evenly over the heads of a group");
  static_assert(GTILE % 1024 == 0, "tiles keep the swizzle alignment");

  // One block's K and V for the head group: one TMA copy each (two per
  // 256-byte-row tile in kWideTwoBoxes mode; see kWideMode).
  __device__ static __forceinline__ void issue(const DecodeArgs &a, uint8_t *sk, int i, int phys, int grp,
                                               uint64_t *bar, uint64_t pol) {
    const int row = (phys * a.num_kv_heads + grp * HG) * 16;
    uint8_t *kd = sk + i * GTILE;
    uint8_t *vd = sk + KVB + i * GTILE;
    if constexpr (ROWB > 128 && kWideMode == kWideHalfMajor) {
      tma_load_3d(kd, &a.kmap, 0, row, 0, bar, pol);
      tma_load_3d(vd, &a.vmap, 0, row, 0, bar, pol);
    } else if constexpr (ROWB > 128 && kWideMode == kWideTokMajor) {
      tma_load_3d(kd, &a.kmap, 0, 0, row, bar, pol);
      tma_load_3d(vd, &a.vmap, 0, 0, row, bar, pol);
    } else if constexpr (ROWB > 128) {
      tma_load_2d(kd, &a.kmap, 0, row, bar, pol);
      tma_load_2d(kd + HG * 16 * 128, &a.kmap, 64, row, bar, pol);
      tma_load_2d(vd, &a.vmap, 0, row, bar, pol);
      tma_load_2d(vd + HG * 16 * 128, &a.vmap, 64, row, bar, pol);
    } else {
      tma_load_2d(kd, &a.kmap, 0, row, bar, pol);
      tma_load_2d(vd, &a.vmap, 0, row, bar, pol);
    }
  }
};

// Merge of a split segment's pieces, run by the epilogue warp of the CTA
// that finished its last piece: CTAs c1..c2 each left a normalised O and an
// lse (log2 domain) per query head in one of their two slots.  out =
// sum_p 2^(lse_p - M) O_p / sum_p 2^(lse_p - M), lse = M + log2(sum), with M
// the largest lse_p.  Slot heads are handled SHC at a time: first one lane
// per (piece, head) for M and the sum, then LPH lanes per head for O.
template <class C>
__device__ void merge_segment(const DecodeArgs &a, const StageHdr &h, long long c1, long long c2, long long per_cta,
                              int lane) {
  constexpr int D = C::D;
  constexpr int GQ = C::GQ;
  constexpr int SH = C::SLOTH;
  constexpr int SHC = SH < 32 ? SH : 32;  // slot heads per pass
  constexpr int PPI = 32 / SHC;           // pieces per lane step of the first loop
  constexpr int LPH = 32 / SHC;           // lanes per head in the second loop
  constexpr int DPL = D / LPH;            // head_dim elements per lane
  constexpr int NF4 = DPL / 4 < 4 ? DPL / 4 : 4;
  static_assert(SH % SHC == 0 && DPL % (4 * NF4) == 0, "merge lane split");
  const int np = static_cast<int>(c2 - c1 + 1);
  auto slot = [&](int p) -> int64_t {
    const long long c = c1 + p;
    return (c * 2 + ((h.seg_start <= c * per_cta) ? 0 : 1)) * SH;
  };
  const int hq0 = h.grp * C::HG * a.g;
  auto qhead = [&](int sj) { return hq0 + (sj / GQ) * a.g + sj % GQ; };
  for (int hb = 0; hb < SH; hb += SHC) {
    // largest lse and sum of 2^(lse - M) per slot head (lane % SHC)
    const int sj = hb + lane % SHC;
    float M = -INFINITY, W = 0.f;
    if (sj % GQ < a.g) {
      for (int p = lane / SHC; p < np; p += PPI) {
        const float x = __ldcg(a.slot_lse + slot(p) + sj);
        if (x == -INFINITY) continue;
        if (x > M) {
          W = W * exp2f(M - x) + 1.f;
          M = x;
        } else {
          W += exp2f(x - M);
        }
      }
    }
#pragma unroll
    for (int o = SHC; o < 32; o <<= 1) {
      const float M2 = __shfl_xor_sync(0xffffffffu, M, o);
      const float W2 = __shfl_xor_sync(0xffffffffu, W, o);
      const float Mn = fmaxf(M, M2);
      W = (M == -INFINITY ? 0.f : W * exp2f(M - Mn)) + (M2 == -INFINITY ? 0.f : W2 * exp2f(M2 - Mn));
      M = Mn;
    }
    if (lane < SHC && sj % GQ < a.g && a.lse)
      a.lse[static_cast<int64_t>(h.s) * a.num_q_heads + qhead(sj)] = M == -INFINITY ? -INFINITY : (M + log2f(W)) * kLn2;
    // weighted sum of the pieces' O: head k of this pass on lanes k * LPH ..
    const int k = lane / LPH;
    const int part = lane % LPH;
    const int sk = hb + k;
    const float Mk = __shfl_sync(0xffffffffu, M, k);
    const float Wk = __shfl_sync(0xffffffffu, W, k);
    if (sk % GQ >= a.g) continue;
    const float inv = Mk == -INFINITY ? 0.f : head_vscale(a, h.grp * C::HG + sk / GQ) / Wk;
    float *o = a.out + (static_cast<int64_t>(h.s) * a.num_q_heads + qhead(sk)) * D + part * DPL;
    for (int f0 = 0; f0 < DPL / 4; f0 += NF4) {
      float4 acc[NF4];
#pragma unroll
      for (int f = 0; f < NF4; ++f) acc[f] = make_float4(0.f, 0.f, 0.f, 0.f);
      if (Mk != -INFINITY) {
#pragma unroll 2
        for (int p = 0; p < np; ++p) {
          const int64_t base = slot(p) + sk;
          const float x = __ldcg(a.slot_lse + base);
          const float4 *src = reinterpret_cast<const float4 *>(a.slot_o + base * D + part * DPL) + f0;
          float4 v[NF4];
#pragma unroll
          for (int f = 0; f < NF4; ++f) v[f] = __ldcg(src + f);
          const float w = x == -INFINITY ? 0.f : exp2f(x - Mk);
#pragma unroll
          for (int f = 0; f < NF4; ++f) {
            acc[f].x += w * v[f].x;
            acc[f].y += w * v[f].y;
            acc[f].z += w * v[f].z;
            acc[f].w += w * v[f].w;
          }
        }
      }
#pragma unroll
      for (int f = 0; f < NF4; ++f)
        reinterpret_cast<float4 *>(o)[f0 + f] =
            make_float4(acc[f].x * inv, acc[f].y * inv, acc[f].z * inv, acc[f].w * inv);
    }
  }
}

// The epilogue warp: folds the consumer warps' partial states of each
// finished piece (per kv head of the group) and writes the output, or this
// CTA's slot when the segment is split across CTAs; the CTA that finishes a
// split segment's last piece merges its pieces (merge_segment).  Runs
// concurrently with the consumers, which move on to the next piece.
template <class C>
__device__ void epilogue(const DecodeArgs &a, const float *red, const StageHdr *rhdr, uint64_t *rfull,
                         uint64_t *rempty, long long per_cta, int lane, int me) {
  constexpr int D = C::D;
  constexpr int NC = C::NC;
  constexpr int HG = C::HG;
  constexpr int BPS = C::BPS;
  constexpr int SH = C::SLOTH;
  int rb = 0;
  uint32_t par = 0;
  for (;;) {
    if (!mbar_wait(&rfull[rb], par, a.wait_ns)) {
      if (lane == 0) report(a, kErrWaitTimeout);
      break;
    }
    const StageHdr h = rhdr[rb];
    if (h.kind == kStageEnd) break;
    const float *R = red + size_t(rb) * NC * C::REDW;
    const long long c1 = h.seg_start / per_cta;
    const long long c2 = (h.seg_start + h.seg_nb - 1) / per_cta;
    const bool split = c1 != c2;
    const int my_slot = (h.seg_start <= static_cast<long long>(me) * per_cta) ? 0 : 1;
    const int hq0 = h.grp * HG * a.g;  // first query head of the group
    for (int hw = 0; hw < HG; ++hw) {
      for (int j = 0; j < a.g; ++j) {
        // warps hw, hw + HG, ... hold this kv head's partials
        float M = -INFINITY;
#pragma unroll
        for (int k = 0; k < BPS; ++k) M = fmaxf(M, R[(hw + HG * k) * C::REDW + j * C::RSTR + D]);
        float cw[BPS];
        float Ls = 0.f;
#pragma unroll
        for (int k = 0; k < BPS; ++k) {
          const float mw = R[(hw + HG * k) * C::REDW + j * C::RSTR + D];
          cw[k] = (mw == -INFINITY) ? 0.f : exp2f(mw - M);
          Ls += R[(hw + HG * k) * C::REDW + j * C::RSTR + D + 1] * cw[k];
        }
        const float inv = 1.f / Ls;
        const float lse2 = M + log2f(Ls);
        const int qh = hq0 + hw * a.g + j;               // query head
        const int sj = hw * C::GQ + j;                   // its place in a slot
        for (int d4 = lane * 4; d4 < D; d4 += 128) {
          float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll
          for (int k = 0; k < BPS; ++k) {
            const float4 v = *reinterpret_cast<const float4 *>(R + (hw + HG * k) * C::REDW + j * C::RSTR + d4);
            acc.x += v.x * cw[k];
            acc.y += v.y * cw[k];
            acc.z += v.z * cw[k];
            acc.w += v.w * cw[k];
          }
          if (!split) {
            const float sc = inv * head_vscale(a, h.grp * HG + hw);
            *reinterpret_cast<float4 *>(a.out + (static_cast<int64_t>(h.s) * a.num_q_heads + qh) * D + d4) =
                make_float4(acc.x * sc, acc.y * sc, acc.z * sc, acc.w * sc);
          } else {
            const int64_t sl = (static_cast<int64_t>(me) * 2 + my_slot) * SH + sj;
            *reinterpret_cast<float4 *>(a.slot_o + sl * D + d4) =
                make_float4(acc.x * inv, acc.y * inv, acc.z * inv, acc.w * inv);
          }
        }
        if (lane == 0) {
          if (!split) {
            if (a.lse) a.lse[static_cast<int64_t>(h.s) * a.num_q_heads + qh] = lse2 * kLn2;
          } else {
            a.slot_lse[(static_cast<int64_t>(me) * 2 + my_slot) * SH + sj] = lse2;
          }
        }
      }
    }
    __syncwarp();
    if (lane == 0) mbar_arrive(&rempty[rb]);
    rb ^= 1;
    if (rb == 0) par ^= 1;
    if (split) {
      // the slot is written; count the piece, and merge if it was the last
      __threadfence();
      __syncwarp();
      int last = 0;
      if (lane == 0) {
        const int seg = h.s * a.num_groups + h.grp;
        const int prev = atom_add_acq_rel_gpu(a.seg_counter + seg, 1);
        last = prev == static_cast<int>(c2 - c1);
        if (last) st_relaxed_gpu(a.seg_counter + seg, 0);  // ready for the next launch
      }
      last = __shfl_sync(0xffffffffu, last, 0);
      __syncwarp();
      if (last) merge_segment<C>(a, h, c1, c2, per_cta, lane);
    }
  }
}

// One partition of the decode work: number me of G equal ranges of the
// flat (segment, block) list (a CTA of the decode kernel, or a work item of
// the mixed-step kernel).  Run by all threads of a CTA; warps past the
// epilogue warp leave after the prologue.  smem_raw: the CTA's dynamic
// shared memory (MmaCfg::SMEM bytes).
template <int D, int KVT, int GQ, int HG, int NS, int NCW>
__device__ void decode_partition(const DecodeArgs &a, uint8_t *smem_raw, int me, int G) {
  using C = MmaCfg<D, KVT, GQ, HG, NS, NCW>;
  constexpr int MT = D / 16;  // m-tiles of O^T (16 head_dim rows each) = k-steps of S^T
  constexpr int NN = C::NN;
  constexpr int NC = C::NC;
  uint8_t *smem = reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint8_t *stages = smem;
  float *red = reinterpret_cast<float *>(smem + size_t(NS) * C::STAGEB);  // [2][NC][GQ][RSTR]
  StageHdr *hdr = reinterpret_cast<StageHdr *>(red + size_t(2) * NC * C::REDW);
  StageHdr *rhdr = hdr + NS;  // [2] piece headers for the epilogue
  uint64_t *full = reinterpret_cast<uint64_t *>(rhdr + 2);
  uint64_t *empty = full + NS;
  uint64_t *rfull = empty + NS;  // [2] partial states ready (NC arrivals)
  uint64_t *rempty = rfull + 2;  // [2] partial states consumed (epilogue)
  __shared__ long long s_per_cta;

  const int tid = threadIdx.x;
  const int warp = tid >> 5;
  const int lane = tid & 31;
  if (tid == 0) {
    for (int i = 0; i < 2; ++i) {
      mbar_init(&rfull[i], NC);
      mbar_init(&rempty[i], 1);
    }
  }
  long long total = 0;
  const long long per_cta = prologue<C>(a, full, empty, &total, &s_per_cta, me, G);
  if (warp == NC) {
    produce<C>(a, stages, hdr, full, empty, per_cta, total, lane, me);
    return;
  }
  if (warp == NC + 1) {
    epilogue<C>(a, red, rhdr, rfull, rempty, per_cta, lane, me);
    return;
  }
  if (warp > NC + 1) return;

  const int hw = warp % HG;  // this warp's kv head within the group
  const int bw = warp / HG;  // and its block within the stage
  const int r = lane >> 2;   // fragment row group
  const int c = lane & 3;    // fragment column pair
  const int lm = lane >> 3;  // ldmatrix: which 8x8 matrix this lane addresses
  const int lr = lane & 7;   // ldmatrix: which row of it
  const int trow = hw * 16;  // first row of this warp's head in a head-group tile
  uint32_t qb[MT][NN][2];    // Q^T B fragments (bf16 or f16 pairs)
  float oacc[MT][NN][4];     // O^T accumulators
  float m[NN][2], l[NN][2];  // per head 2c, 2c+1 of each n-tile
#pragma unroll
  for (int nn = 0; nn < NN; ++nn) {
    m[nn][0] = m[nn][1] = -INFINITY;
    l[nn][0] = l[nn][1] = 0.f;
#pragma unroll
    for (int mt = 0; mt < MT; ++mt) oacc[mt][nn][0] = oacc[mt][nn][1] = oacc[mt][nn][2] = oacc[mt][nn][3] = 0.f;
  }
  int stage = 0;
  uint32_t cpar = 0;
  int rb = 0;
  uint32_t rpar = 1;  // the partial-state buffers start out free
  float qsc = a.qscale;  // score scale of this warp's kv head (set per segment)
  // pa_decode_append: this lane's 16-byte chunk of the segment's appended K
  // (lanes < ROWB / 16) or V row, and its byte offset in the cache (-1: none)
  uint4 app = make_uint4(0, 0, 0, 0);
  int64_t app_off = -1;
  PA_TRACE(const long long tc0 = clock64(); long long tc_full = 0, tc_fin = 0, n_st = 0, n_pc = 0;)
  for (;;) {
    PA_TRACE(const long long tw0 = clock64();)
    if (!mbar_wait(&full[stage], cpar, a.wait_ns)) {
      if (lane == 0) report(a, kErrWaitTimeout);
      break;
    }
    PA_TRACE(tc_full += clock64() - tw0; ++n_st;)
    const StageHdr h = hdr[stage];
    if (h.kind == kStageEnd) break;
    const uint8_t *Ks = stages + size_t(stage) * C::STAGEB;
    const uint8_t *Vs = Ks + C::KVB;
    if (h.flags & kFlagFirst) {
      qsc = head_qscale(a, h.grp * HG + hw);
      {
        if (a.k_new != nullptr && lane < 2 * (C::ROWB / 16)) {
          // the token this step appends to the sequence (position L - 1),
          // loaded now so that the sequence's last block finds it in
          // registers: a 16-byte chunk of its cache row (K for lanes < CH,
          // else V) and where it goes in the cache
          constexpr int CH = C::ROWB / 16;
          const int kvh = h.grp * HG + hw;
          const int ch = lane % CH;
          const bool is_k = lane < CH;
          const uint8_t *src = is_k ? a.k_new : a.v_new;
          const int64_t row = static_cast<int64_t>(h.s) * a.num_kv_heads + kvh;
          if constexpr (kv16(KVT)) {
            app = __ldg(reinterpret_cast<const uint4 *>(src + row * C::ROWB) + ch);
          } else {
            // 16 activation values (32 bytes) become 16 cache bytes
            const uint4 *s2 = reinterpret_cast<const uint4 *>(src + row * (2 * C::ROWB)) + 2 * ch;
            const float *hs = is_k ? a.k_scales : a.v_scales;
            const float sc = hs ? __ldg(hs + kvh) : (is_k ? a.k_enc : a.v_enc);
            app = encode_fp8x16<KVT>(__ldg(s2), __ldg(s2 + 1), sc);
          }
          const int L = seq_len(a, h.s);
          app_off = -1;
          if (L > 0) {
            const int phys = __ldg(a.block_tables + static_cast<int64_t>(h.s) * a.max_blocks_per_seq + ((L - 1) >> 4));
            if (!a.checked || (phys >= 0 && phys < a.num_blocks))
              app_off = ((static_cast<int64_t>(phys) * a.num_kv_heads + kvh) * 16 + ((L - 1) & 15)) * C::ROWB + ch * 16;
            else
              report(a, kErrBadIndex);  // no row is written outside the cache
          }
        }
      }
      // Q^T fragments of this kv head's query heads (zero past g)
      const uint16_t *Qs = reinterpret_cast<const uint16_t *>(Ks + C::QOFF) + hw * a.g * D;
#pragma unroll
      for (int nn = 0; nn < NN; ++nn) {
        const int n = nn * 8 + r;
        const bool hv = n < a.g;
#pragma unroll
        for (int ks = 0; ks < MT; ++ks) {
          if constexpr (kv16(KVT)) {
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
    const int vt = h.ntok - 16 * bw;  // valid tokens of this warp's block (<= 0: none)
    if (vt > 0) {
      {
        if (a.k_new != nullptr && (h.flags & kFlagEnd) && vt <= 16) {
          // the sequence's last block: its row vt - 1 is the appended token,
          // put into the staged tile (over the cache's stale row) before any
          // fragment of the block is read, and into the cache
          constexpr int CH = C::ROWB / 16;
          if (lane < 2 * CH) {
            uint8_t *tile = const_cast<uint8_t *>(lane < CH ? Ks : Vs) + bw * C::GTILE;
            *reinterpret_cast<uint4 *>(tile + swz_off<C::ROWB, HG>(trow + vt - 1, lane % CH)) = app;
            if (app_off >= 0) *reinterpret_cast<uint4 *>((lane < CH ? a.k_write : a.v_write) + app_off) = app;
          }
          fence_proxy_async_smem();  // the stage's next copy lands after these writes
          __syncwarp();
        }
      }
      const uint32_t kt = smem_u32(Ks + bw * C::GTILE);
      const uint32_t vtl = smem_u32(Vs + bw * C::GTILE);
      // ---- S^T (16 tokens x 8 heads per n-tile) = K Q^T, two accumulator
      // chains (even and odd k-steps)
      float sa[NN][4], sb[NN][4];
#pragma unroll
      for (int nn = 0; nn < NN; ++nn)
#pragma unroll
        for (int e = 0; e < 4; ++e) sa[nn][e] = sb[nn][e] = 0.f;
      if constexpr (kv16(KVT)) {
#pragma unroll
        for (int ks = 0; ks < MT; ++ks) {
          uint32_t a0, a1, a2, a3;
          ldmatrix_x4(a0, a1, a2, a3, kt + swz_off<C::ROWB, HG>(trow + lr + (lm & 1) * 8, 2 * ks + (lm >> 1)));
#pragma unroll
          for (int nn = 0; nn < NN; ++nn) {
            if (ks & 1)
              mma16_16816<KVT>(sb[nn], a0, a1, a2, a3, qb[ks][nn][0], qb[ks][nn][1]);
            else
              mma16_16816<KVT>(sa[nn], a0, a1, a2, a3, qb[ks][nn][0], qb[ks][nn][1]);
          }
        }
      } else {
#pragma unroll
        for (int j = 0; j < MT; j += 2) {
          uint32_t r0, r1, r2, r3;
          ldmatrix_x4(r0, r1, r2, r3, kt + swz_off<C::ROWB, HG>(trow + lr + (lm & 1) * 8, j + (lm >> 1)));
          const uint32_t a0 = fp8x2_to_f16x2<KVT>(static_cast<uint16_t>(r0 & 0xffffu));
          const uint32_t a2 = fp8x2_to_f16x2<KVT>(static_cast<uint16_t>(r0 >> 16));
          const uint32_t a1 = fp8x2_to_f16x2<KVT>(static_cast<uint16_t>(r1 & 0xffffu));
          const uint32_t a3 = fp8x2_to_f16x2<KVT>(static_cast<uint16_t>(r1 >> 16));
          const uint32_t b0 = fp8x2_to_f16x2<KVT>(static_cast<uint16_t>(r2 & 0xffffu));
          const uint32_t b2 = fp8x2_to_f16x2<KVT>(static_cast<uint16_t>(r2 >> 16));
          const uint32_t b1 = fp8x2_to_f16x2<KVT>(static_cast<uint16_t>(r3 & 0xffffu));
          const uint32_t b3 = fp8x2_to_f16x2<KVT>(static_cast<uint16_t>(r3 >> 16));
#pragma unroll
          for (int nn = 0; nn < NN; ++nn) {
            mma_f16_16816(sa[nn], a0, a1, a2, a3, qb[j][nn][0], qb[j][nn][1]);
            mma_f16_16816(sb[nn], b0, b1, b2, b3, qb[j + 1][nn][0], qb[j + 1][nn][1]);
          }
        }
      }
      // ---- online softmax over the block's tokens, per head (column)
      uint32_t pb[NN][2], pbl[NN][2];
      // tokens of this warp's block before the first key (local attention)
      // or past the sequence's end are out
      const int vl = h.tlo - 16 * bw;
      const bool v_lo = r < vt && r >= vl, v_hi = r + 8 < vt && r + 8 >= vl;
#pragma unroll
      for (int nn = 0; nn < NN; ++nn) {
        const float s0 = v_lo ? (sa[nn][0] + sb[nn][0]) * qsc : -INFINITY;
        const float s1 = v_lo ? (sa[nn][1] + sb[nn][1]) * qsc : -INFINITY;
        const float s2 = v_hi ? (sa[nn][2] + sb[nn][2]) * qsc : -INFINITY;
        const float s3 = v_hi ? (sa[nn][3] + sb[nn][3]) * qsc : -INFINITY;
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
        if constexpr (kv16(KVT)) {
          // P as a hi + lo pair of the cache's 16-bit type
          const uint32_t h01 = pack16x2<KVT>(p0, p1), h23 = pack16x2<KVT>(p2, p3);
          pb[nn][0] = movmatrix_trans(h01);
          pb[nn][1] = movmatrix_trans(h23);
          pbl[nn][0] = movmatrix_trans(pack16x2<KVT>(p0 - lo16<KVT>(h01), p1 - hi16<KVT>(h01)));
          pbl[nn][1] = movmatrix_trans(pack16x2<KVT>(p2 - lo16<KVT>(h23), p3 - hi16<KVT>(h23)));
        } else {
          pb[nn][0] = movmatrix_trans(pack_f16x2(p0, p1));
          pb[nn][1] = movmatrix_trans(pack_f16x2(p2, p3));
        }
      }
      // ---- O^T += V^T P^T.  Tokens outside the block's valid range may hold
      // anything (NaN included); a zero probability does not cancel them
      // (0 * NaN = NaN), so their V^T fragment entries are zeroed: mk_lo
      // covers tokens 2c, 2c+1 and mk_hi tokens 2c+8, 2c+9 of this lane.
      auto in = [&](int t) { return t < vt && t >= vl; };
      const uint32_t mk_lo = (in(2 * c) ? 0x0000ffffu : 0u) | (in(2 * c + 1) ? 0xffff0000u : 0u);
      const uint32_t mk_hi = (in(2 * c + 8) ? 0x0000ffffu : 0u) | (in(2 * c + 9) ? 0xffff0000u : 0u);
      if constexpr (kv16(KVT)) {
#pragma unroll
        for (int mt = 0; mt < MT; ++mt) {
          uint32_t a0, a1, a2, a3;
          ldmatrix_x4_trans(a0, a1, a2, a3, vtl + swz_off<C::ROWB, HG>(trow + lr + (lm >> 1) * 8, 2 * mt + (lm & 1)));
          a0 &= mk_lo;
          a1 &= mk_lo;
          a2 &= mk_hi;
          a3 &= mk_hi;
#pragma unroll
          for (int nn = 0; nn < NN; ++nn) {
            mma16_16816<KVT>(oacc[mt][nn], a0, a1, a2, a3, pb[nn][0], pb[nn][1]);
            mma16_16816<KVT>(oacc[mt][nn], a0, a1, a2, a3, pbl[nn][0], pbl[nn][1]);
          }
        }
      } else {
#pragma unroll
        for (int j = 0; j < MT; j += 2) {
          uint32_t r0, r1, r2, r3;
          ldmatrix_x4_trans(r0, r1, r2, r3, vtl + swz_off<C::ROWB, HG>(trow + lr + (lm & 1) * 8, j + (lm >> 1)));
          // r0: tokens 2c, 2c+1 (of 0-7) x d = 16j + 2r, 2r+1 as bytes
          // (t,d), (t,d+1), (t+1,d), (t+1,d+1); the permute pairs the tokens
          const uint32_t x0 = __byte_perm(r0, 0, 0x3120), x1 = __byte_perm(r1, 0, 0x3120);
          const uint32_t y0 = __byte_perm(r2, 0, 0x3120), y1 = __byte_perm(r3, 0, 0x3120);
          const uint32_t a0 = fp8x2_to_f16x2<KVT>(static_cast<uint16_t>(x0 & 0xffffu)) & mk_lo;
          const uint32_t a1 = fp8x2_to_f16x2<KVT>(static_cast<uint16_t>(x0 >> 16)) & mk_lo;
          const uint32_t a2 = fp8x2_to_f16x2<KVT>(static_cast<uint16_t>(x1 & 0xffffu)) & mk_hi;
          const uint32_t a3 = fp8x2_to_f16x2<KVT>(static_cast<uint16_t>(x1 >> 16)) & mk_hi;
          const uint32_t b0 = fp8x2_to_f16x2<KVT>(static_cast<uint16_t>(y0 & 0xffffu)) & mk_lo;
          const uint32_t b1 = fp8x2_to_f16x2<KVT>(static_cast<uint16_t>(y0 >> 16)) & mk_lo;
          const uint32_t b2 = fp8x2_to_f16x2<KVT>(static_cast<uint16_t>(y1 & 0xffffu)) & mk_hi;
          const uint32_t b3 = fp8x2_to_f16x2<KVT>(static_cast<uint16_t>(y1 >> 16)) & mk_hi;
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
    PA_TRACE(const long long tf0 = clock64(); ++n_pc;)

    // ---- hand this warp's partial state of the piece to the epilogue warp
#pragma unroll
    for (int nn = 0; nn < NN; ++nn)
#pragma unroll
      for (int e = 0; e < 2; ++e)
#pragma unroll
        for (int o = 4; o < 32; o <<= 1) l[nn][e] += __shfl_xor_sync(0xffffffffu, l[nn][e], o);
    if (!mbar_wait(&rempty[rb], rpar, a.wait_ns)) {
      if (lane == 0) report(a, kErrWaitTimeout);
      break;
    }
    float *rw = red + (size_t(rb) * NC + warp) * C::REDW;
#pragma unroll
    for (int nn = 0; nn < NN; ++nn) {
      const int h0 = nn * 8 + 2 * c;
      if (h0 < GQ) {
        if (r == 0) {
          rw[h0 * C::RSTR + D] = m[nn][0];
          rw[h0 * C::RSTR + D + 1] = l[nn][0];
          rw[(h0 + 1) * C::RSTR + D] = m[nn][1];
          rw[(h0 + 1) * C::RSTR + D + 1] = l[nn][1];
        }
#pragma unroll
        for (int mt = 0; mt < MT; ++mt) {
          // bf16: rows r, r+8 of m-tile mt are d = 16mt + r, 16mt + 8 + r;
          // E4M3: d = 16mt + 2r, 16mt + 2r + 1
          const int dlo = kv16(KVT) ? mt * 16 + r : mt * 16 + 2 * r;
          const int dhi = kv16(KVT) ? dlo + 8 : dlo + 1;
          rw[h0 * C::RSTR + dlo] = oacc[mt][nn][0];
          rw[(h0 + 1) * C::RSTR + dlo] = oacc[mt][nn][1];
          rw[h0 * C::RSTR + dhi] = oacc[mt][nn][2];
          rw[(h0 + 1) * C::RSTR + dhi] = oacc[mt][nn][3];
        }
      }
    }
    if (warp == 0 && lane == 0) rhdr[rb] = h;
    __syncwarp();
    if (lane == 0) mbar_arrive(&rfull[rb]);
    rb ^= 1;
    if (rb == 0) rpar ^= 1;
    PA_TRACE(tc_fin += clock64() - tf0;)
  }
  // tell the epilogue warp that no piece follows
  if (mbar_wait(&rempty[rb], rpar, a.wait_ns)) {
    if (warp == 0 && lane == 0) rhdr[rb].kind = kStageEnd;
    __syncwarp();
    if (lane == 0) mbar_arrive(&rfull[rb]);
  } else if (lane == 0) {
    report(a, kErrWaitTimeout);
  }
  PA_TRACE(if (tid == 0) {
    g_pa_trace[me][0] = tc_full;
    g_pa_trace[me][1] = tc_fin;
    g_pa_trace[me][2] = clock64() - tc0;
    g_pa_trace[me][6] = n_st;
    g_pa_trace[me][7] = n_pc;
  })
}

template <int D, int KVT, int GQ, int HG, int NS, int NCW>
__global__ void __launch_bounds__((NCW + 2) * 32, 1) decode_mma_kernel(const __grid_constant__ DecodeArgs a) {
  // launched as a programmatic dependent of the preceding kernel in the
  // stream: nothing is read before that kernel's writes are visible.  (No
  // early launch_dependents: CTAs of a following grid parked on the SMs
  // while this one drains measured 0.2-0.9 us slower per launch.)
  asm volatile("griddepcontrol.wait;" ::: "memory");
  extern __shared__ uint8_t smem_raw[];
  decode_partition<D, KVT, GQ, HG, NS, NCW>(a, smem_raw, blockIdx.x, gridDim.x);
}

// ------------------------------------------------------------ kernel lookup

// A decode kernel instantiation and what the host needs to launch it.
struct KernelInfo {
  void *fn = nullptr;
  size_t smem = 0;
  int threads = 0;
  int slot_heads = 0;  // query heads of one slot (HG x padded group)
  int hg = 1;          // kv heads per stage group
  bool mma = false;
  int swizzle = 0;     // MMA: 128 or 64 byte TMA swizzle
  int wide_mode = 0;   // MMA: copy shape of 256-byte rows (kWide*)
};

// SIMT: stages of about 32 KB, three of them, two CTAs per SM
template <int D, int KVT, int GP>
KernelInfo simt_info() {
  constexpr int ESZ = kv16(KVT) ? 2 : 1;
  constexpr int BPS = (D * ESZ >= 256) ? 4 : 8;
  using Cfg = SimtCfg<D, KVT, GP, BPS, 3>;
  KernelInfo k;
  k.fn = reinterpret_cast<void *>(&decode_simt_kernel<D, KVT, GP, BPS, 3>);
  k.smem = Cfg::SMEM;
  k.threads = Cfg::NTHREADS;
  k.slot_heads = Cfg::SLOTH;
  k.hg = 1;
  return k;
}

// MMA: as many stages as fit next to the partial-state buffers in about
// 220 KB of shared memory (at most 12), one CTA per SM.  NCW consumer warps:
// 4 suffice to keep up with the bf16 stream; the E4M3 consumers also
// convert every element (about one instruction per KV byte) and need 8, two
// per SM sub-partition, to hide each other's latency (measured on GB300:
// 67% -> 89% of the HBM copy rate).
template <int D, int KVT, int GQ, int HG, int NCW = kConsumerWarps>
constexpr int mma_stages() {
  constexpr int ESZ = kv16(KVT) ? 2 : 1;
  constexpr int STAGEB = 2 * NCW * 16 * D * ESZ + ((HG * GQ * D * 2 + 1023) / 1024) * 1024;
  constexpr int RED = 2 * NCW * GQ * (D + 4) * 4;
  constexpr int FIT = (225280 - 2048 - RED) / STAGEB;
  return FIT > 12 ? 12 : FIT;
}

template <int D, int KVT, int GQ, int HG, int NCW = kConsumerWarps>
KernelInfo mma_info() {
  constexpr int NS = mma_stages<D, KVT, GQ, HG, NCW>();
  static_assert(NS >= 3, "at least three stages in flight");
  using Cfg = MmaCfg<D, KVT, GQ, HG, NS, NCW>;
  KernelInfo k;
  k.fn = reinterpret_cast<void *>(&decode_mma_kernel<D, KVT, GQ, HG, NS, NCW>);
  k.smem = Cfg::SMEM;
  k.threads = Cfg::NTHREADS;
  k.slot_heads = Cfg::SLOTH;
  k.hg = HG;
  k.mma = true;
  k.swizzle = Cfg::ROWB >= 128 ? 128 : 64;
  k.wide_mode = kWideMode;
  return k;
}

// 8-bit caches (E4M3 or E5M2, per KVT): 8 consumer warps (see mma_info)
// while their partial-state buffers leave room for enough stages (up to 8
// query heads per kv head), else 4; kv-head groups of 2 or 1.
template <int GQ>
constexpr int fp8_consumer_warps() {
  return GQ <= 8 ? 8 : 4;
}

template <int KVT, int D, int GQ>
KernelInfo fp8_mma_for_hg(int hg) {
  if (hg >= 2) return mma_info<D, KVT, GQ, 2, fp8_consumer_warps<GQ>()>();
  return mma_info<D, KVT, GQ, 1, fp8_consumer_warps<GQ>()>();
}

template <int KVT, int D>
KernelInfo fp8_mma_for(int gq, int hg) {
  if (gq <= 4) return fp8_mma_for_hg<KVT, D, 4>(hg);
  if (gq <= 8) return fp8_mma_for_hg<KVT, D, 8>(hg);
  return fp8_mma_for_hg<KVT, D, 16>(hg);
}

// The kernel arguments of a decode call planned as `plan` (tensor maps for
// the MMA kernel); false if a tensor map cannot be made.  pa_decode.cu.
bool make_decode_args(const pa_kv_desc &d, const DecodePlan &plan, float *out, float *lse, const void *q,
                      const void *k_cache, const void *v_cache, const int32_t *block_tables,
                      int32_t max_blocks_per_seq, const int32_t *context_lens, int32_t num_seqs, float scale,
                      void *workspace, DecodeArgs *a);

// Defined in the translation units that instantiate the kernels.
KernelInfo pick_simt(int head_dim, int kv_dtype, int g);
KernelInfo pick_mma_bf16(int head_dim, int gq, int hg);
KernelInfo pick_mma_f16(int head_dim, int gq, int hg);
KernelInfo pick_mma_fp8(int head_dim, int gq, int hg);   // E4M3
KernelInfo pick_mma_e5m2(int head_dim, int gq, int hg);

}  // namespace dec
}  // namespace pa
