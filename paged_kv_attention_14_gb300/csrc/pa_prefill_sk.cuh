// pa_prefill_sk.cuh -- the balanced tcgen05 chunked prefill
// (pa_prefill_chunk_balanced): what pa_prefill_tc.cuh computes, with the
// work of all items spread evenly over one CTA per SM.
//
// Why: the grid kernel gives each item (256 query-head rows of one sequence
// and kv head: a "chunked prefill" chunk's query tile, vllm.cpp
// implementation notes, Engine core bullet) its own CTA.  n items of similar
// length run in ceil(n / SMs) waves, and the last wave may leave SMs idle.
//
// How (GB300 design):
//  * A unit is one 128-key KV tile of one item.  Items are ordered by kv
//    head, then pair (sequence, query tile); CTA c of G takes units
//    [c U / G, (c + 1) U / G) (a stream-K decomposition).  An item whose
//    units fall to several CTAs is computed in pieces.  Each piece leaves its
//    normalised output and log-sum-exp in a slot of the workspace; the CTA
//    that finishes the last piece merges them all by log-sum-exp once its
//    own pipeline has drained.
//  * Each CTA runs its items ("segments") as one continuous pipeline.  The
//    K/V rings and every barrier keep counting across segments.  The
//    producer loads a segment's first K tiles while the previous one is
//    still computing, and its Q once that segment's last QKs completed
//    (Q_EMPTY).  The MMA issuer goes straight from a segment's last P.V to
//    the next segment's first QKs, and the softmax warps write a segment's
//    output while the tensor cores start on the next.  The next segment's
//    first P.V overwrites O only after the softmax's arrival for its scores,
//    which follows the reads of the previous O.
//  * Roles and tiles are those of the grid kernel (see pa_prefill_tc.cuh):
//    warp 0 MMA issuer, warp 1 TMA producer (and the thread-staged Q tiles),
//    warps 2-3 K / V preparation, warps 4-11 the softmax.
#pragma once

#include "pa_prefill_tc.cuh"

namespace pa {
namespace pftc {

// One CTA's segments, in the order it runs them: the range's last item
// first when it runs on into the next CTA and is not also the range's first
// (the neighbour starts its own piece of that item at once, so both pieces
// of the item are in flight together), then the range from its first unit.
// Units are ordered by kv head, then pair (sequence, query tile), then
// iteration, so that neighbouring CTAs read the same sequence's K/V of one
// kv head at about the same time.  Every thread of the CTA walks its own
// copy; all copies yield the same segments.
struct SkIter {
  int u, ub;  // walk: next unit, end (the range's end, or zs)
  int u1;     // the range's end
  int base;   // the first unit of item (p, kvh)
  int zs;     // the first unit of the item run first
  int U;      // units of the launch (the host keeps it below 2^31)
  int T;      // units per kv head (all pairs' iterations)
  int p, np, kvh, it;  // walk: pair, its iterations, kv head, iteration
  int pz, nz, kvz;     // the item run first: pair, iterations, kv head
  int z_first;         // it is still to run
  int G, me, H, P;

  __device__ __forceinline__ bool more() const { return z_first || u < ub; }

  __device__ __forceinline__ void fill(const Args &a, Seg &sg, int pp, int start, int n, int kv, int lo,
                                       int hi) const {
    sg.s = pp / a.gx;
    sg.split = 0;
    sg.kvh = kv;
    sg.qtile = a.gx - 1 - pp % a.gx;
    sg.gx = a.gx;
    sg.it_lo = lo;
    sg.it_hi = hi;
    sg.item_start = start;
    sg.U = U;
    sg.G = G;
    sg.me = me;
    sg.c_lo = sk_cta_of(start, U, G);
    sg.c_hi = sk_cta_of(start + n - 1, U, G);
    sg.piece = sg.c_lo != sg.c_hi;
    sg.slot = sk_slot(me, start, U, G);
    sg.item = pp * H + kv;
  }

  // The next segment; false after the last.
  __device__ __forceinline__ bool next(const Args &a, Seg &sg) {
    if (z_first) {
      // the piece [zs, u1) of the item that runs on into the next CTA
      z_first = 0;
      fill(a, sg, pz, zs, nz, kvz, 0, u1 - zs);
      return true;
    }
    if (u >= ub) return false;
    const int len = min(np - it, ub - u);
    fill(a, sg, p, base, np, kvh, it, it + len);
    const bool done = it + len == np;  // the item is finished
    u += len;
    it = 0;
    if (u < ub && done) {
      base += np;
      do {
        if (++p == P) {
          p = 0;
          ++kvh;
        }
        np = pair_iters(a, p);
      } while (np == 0);
    }
    return true;
  }
};

// A merge a CTA owes: it finished the last piece of a cut item.  The item's
// pieces lie in the slots of CTAs c_lo .. c_hi; its rows are those of
// sequence rows qs + qt0 .. (nq queries) and kv head kvh.
struct SkMerge {
  int item_start, c_lo, c_hi, qs, qt0, nq, kvh;
  float vscale;
};
constexpr int kMaxMerges = 2;  // a CTA's first and last items are its only pieces
static_assert(16 + kMaxMerges * sizeof(SkMerge) <= 128, "merge list fits its 128 bytes");

// The merges a CTA owes, once its pipeline has drained (every copy and
// product complete, the rings free):
//   out = sum_c w_c O_c / sum_c w_c,  w_c = 2^(lse_c - M),  M = max_c lse_c,
//   lse = M + log2(sum_c w_c)  (in natural-log units on output)
// over the item's pieces in CTA order (the log-sum-exp combination of
// partial softmax results, as pa_merge_partials computes it; the bits do not
// depend on which piece finished last).  Per Q tile, each piece's 64 KB of
// partial output comes into shared memory by one bulk copy, two buffers
// deep, and softmax thread (row r, half h) accumulates its half of row r.
template <int D, int KVT, int PVM>
__device__ void sk_run_merges(const Args &a, uint8_t *smem, int U, int G, int nmerge) {
  using C = Cfg<D, KVT, PVM>;
  uint64_t *bar = reinterpret_cast<uint64_t *>(smem + C::OFF_BAR);
  const SkMerge *ml = reinterpret_cast<const SkMerge *>(smem + C::OFF_M + 16);
  constexpr int TB = MT * D * 4;  // one Q tile of a piece
  static_assert(2 * TB < C::OFF_BAR - C::OFF_K, "two tile buffers fit the K and V rings");
  uint8_t *buf0 = smem + C::OFF_K;
  // the pieces' log-sum-exp vectors (MROWS floats each) behind the buffers
  float *lse_s = reinterpret_cast<float *>(smem + C::OFF_K + 2 * TB);
  constexpr int kLseCap = (C::OFF_BAR - C::OFF_K - 2 * TB) / (MROWS * 4);
  const int tid = threadIdx.x;
  const int warp = tid >> 5;
  const int lane = tid & 31;
  const bool mt = warp >= kSoftmaxWarp0;  // the merging threads
  const int h = (warp - kSoftmaxWarp0) >> 2;
  const int r = ((warp & 3) << 5) | lane;
  const int g = a.g;
  const int rows_used = a.qt * g;
  if (tid == 0) {
    mbar_init(&bar[K_FULL], 1);      // tile buffer 0
    mbar_init(&bar[K_FULL + 1], 1);  // tile buffer 1
    mbar_init(&bar[V_FULL], 1);      // the log-sum-exp vectors
    fence_mbar_init();
  }
  __syncthreads();
  bool ok = true;
  int q = 0;  // tile copies issued so far (buffer q & 1, its barrier's phase (q >> 1) & 1)
  auto issue = [&](int qq, const SkMerge &m, int c, int t) {
    const int64_t sl = sk_slot(c, m.item_start, U, G);
    fence_proxy_async_smem();  // earlier reads of the buffer precede the copy's writes
    mbar_arrive_expect_tx(&bar[K_FULL + (qq & 1)], TB);
    bulk_g2s(buf0 + (qq & 1) * TB, a.part_o + (sl * NQT + t) * (D / 4) * MT * 4, TB, &bar[K_FULL + (qq & 1)]);
  };
  for (int e = 0; e < nmerge; ++e) {
    const SkMerge m = ml[e];
    const int n = m.c_hi - m.c_lo + 1;
    // the pieces' log-sum-exp vectors: into shared memory by one bulk copy
    // each (1 KB), or read from global memory where more pieces than fit
    const bool lse_smem = n <= kLseCap;
    if (tid == 0 && lse_smem) {
      fence_proxy_async_smem();
      mbar_arrive_expect_tx(&bar[V_FULL], n * MROWS * 4);
      for (int c = m.c_lo; c <= m.c_hi; ++c)
        bulk_g2s(lse_s + (c - m.c_lo) * MROWS, a.part_lse + static_cast<int64_t>(sk_slot(c, m.item_start, U, G)) * MROWS,
                 MROWS * 4, &bar[V_FULL]);
    }
    if (lse_smem && !mbar_wait(&bar[V_FULL], e & 1, a.wait_ns)) ok = false;
    auto lse_of = [&](int c, int R) {
      return lse_smem ? lse_s[(c - m.c_lo) * MROWS + R]
                      : __ldcg(a.part_lse + static_cast<int64_t>(sk_slot(c, m.item_start, U, G)) * MROWS + R);
    };
    for (int t = 0; t < NQT; ++t) {
      const int R = t * MT + r;
      const int qi = R / g;
      const bool rv = mt && ok && R < rows_used && qi < m.nq;
      if (tid == 0) issue(q, m, m.c_lo, t);
      float M = -INFINITY, W = 0.f;
      if (rv) {
        for (int c = m.c_lo; c <= m.c_hi; ++c) M = fmaxf(M, lse_of(c, R));
        if (M == -INFINITY) M = 0.f;  // no key in any piece: every weight is 0
        for (int c = m.c_lo; c <= m.c_hi; ++c) W += exp2f(lse_of(c, R) - M);
      }
      float acc[D / 2];
#pragma unroll
      for (int i = 0; i < D / 2; ++i) acc[i] = 0.f;
      for (int c = m.c_lo; c <= m.c_hi; ++c, ++q) {
        if (tid == 0 && c < m.c_hi) issue(q + 1, m, c + 1, t);
        if (mt) {
          const float w = rv ? exp2f(lse_of(c, R) - M) : 0.f;
          if (!mbar_wait(&bar[K_FULL + (q & 1)], (q >> 1) & 1, a.wait_ns)) ok = false;
          if (ok && rv) {
            const float4 *x = reinterpret_cast<const float4 *>(buf0 + (q & 1) * TB);
#pragma unroll
            for (int k = 0; k < D / 8; ++k) {
              const float4 y = x[(h * (D / 8) + k) * MT + r];
              acc[4 * k] = __fmaf_rn(w, y.x, acc[4 * k]);
              acc[4 * k + 1] = __fmaf_rn(w, y.y, acc[4 * k + 1]);
              acc[4 * k + 2] = __fmaf_rn(w, y.z, acc[4 * k + 2]);
              acc[4 * k + 3] = __fmaf_rn(w, y.w, acc[4 * k + 3]);
            }
          }
        }
        __syncthreads();  // the buffer is read: the copy after next may replace it
      }
      if (rv && ok) {
        const float sc = W > 0.f ? m.vscale / W : 0.f;
        const int64_t orow_i = static_cast<int64_t>(m.qs + m.qt0 + qi) * a.num_q_heads + m.kvh * g + (R - qi * g);
        float *orow = a.out + orow_i * D + h * (D / 2);
#pragma unroll
        for (int i = 0; i < D / 2; i += 4)
          *reinterpret_cast<float4 *>(orow + i) = make_float4(acc[i] * sc, acc[i + 1] * sc, acc[i + 2] * sc, acc[i + 3] * sc);
        if (h == 0 && a.lse) a.lse[orow_i] = W > 0.f ? (M + log2f(W)) * kLn2 : -INFINITY;
      }
    }
    __syncthreads();  // every read of the log-sum-exp vectors is done before the next merge's copies
  }
  // a wait that ran out: the copies still in flight land before the CTA exits
  if (!__syncthreads_and(ok)) {
    if (tid == 0) {
      report_error(a.err, a.ws_err, kErrWaitTimeout);
      for (int i = max(0, q - 2); i < q; ++i) mbar_wait(&bar[K_FULL + (i & 1)], (i >> 1) & 1, a.wait_ns);
      mbar_wait(&bar[V_FULL], (nmerge - 1) & 1, a.wait_ns);
    }
    __syncthreads();
  }
}

// The continuous pipeline of one CTA over its segments.  Run by all
// NTHREADS threads with tensor memory allocated; on return every copy and
// product has completed.  Per-segment phases: Q_FULL and Q_EMPTY complete
// once per segment; K/V ring slots, S_FULL and P_FULL once per KV iteration
// counted over all segments (git); S_FULL_t completes once more after the
// last iteration (O_t final).
template <int D, int KVT, int PVM>
__device__ void prefill_run(const Args &a, uint8_t *smem, uint32_t tmem, const SkIter &it0) {
  using C = Cfg<D, KVT, PVM>;
  uint64_t *bar = reinterpret_cast<uint64_t *>(smem + C::OFF_BAR);
  uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(bar + NBAR);
  int *s_abort = reinterpret_cast<int *>(tmem_slot + 1);
  int *s_last_k = s_abort + 1;  // last KV iteration whose K copies the producer issued
  int *s_last_v = s_abort + 2;  // ... and whose V copies
  int *s_last_q = s_abort + 4;  // last segment whose Q tiles the producer copied by TMA
  const int tid = threadIdx.x;
  const int warp = tid >> 5;
  const int lane = tid & 31;
  const int g = a.g;
  const int rows_used = a.qt * g;

  if (tid == 0) {
    for (int i = 0; i < NSK; ++i) {
      mbar_init(&bar[K_FULL + i], 1);
      mbar_init(&bar[K_EMPTY + i], 1);
      mbar_init(&bar[K_READY + i], 2);
    }
    for (int i = 0; i < NSV; ++i) {
      mbar_init(&bar[V_FULL + i], 1);
      mbar_init(&bar[V_EMPTY + i], 1);
      mbar_init(&bar[V_READY + i], 2);
    }
    for (int t = 0; t < NQT; ++t) {
      mbar_init(&bar[S_FULL + t], 1);
      mbar_init(&bar[P_FULL + t], 8);
    }
    mbar_init(&bar[Q_FULL], 1);
    mbar_init(&bar[Q_EMPTY], 1);
    *s_abort = 0;
    *s_last_k = -1;
    *s_last_v = -1;
    *s_last_q = -1;
    *reinterpret_cast<int *>(smem + C::OFF_M) = 0;  // merges owed
    fence_mbar_init();
  }
  tc_fence_before_sync();
  __syncthreads();
  tc_fence_after_sync();
  const uint32_t sbase = smem_u32(smem);

  if (warp == kProducerWarp) {
    // ------------------------------------------------------ TMA producer
    // per segment: K of its first tile, then its Q (once the previous
    // segment's last QKs completed), then V of the first tile and the rest
    const uint64_t pol = l2_evict_first_policy();
    constexpr int BOXES = C::KV8 ? 1 : C::HALVES;
    const int bi = lane / BOXES;
    const int hh = lane % BOXES;
    const bool issuer = lane < BPT * BOXES;
    SkIter iter = it0;
    Seg sg;
    bool ok = true;
    int git = 0;
    // test hook: issue nothing and signal nothing, so the other warps' waits
    // run out with nothing in flight
    for (int k = 0; ok && !a.stall && iter.next(a, sg); ++k) {
      ItemRange ir;
      item_range(a, sg.s, 0, sg.qtile, sg.gx, true, ir);
      const int32_t *table = a.block_tables + static_cast<int64_t>(sg.s) * a.max_blocks_per_seq;
      auto block_id = [&](int lb) {
        const int v = __ldg(table + lb);
        return a.checked ? checked_block(v, a.num_blocks, a.err, a.ws_err) : v;
      };
      const int kv_lo = ir.kv_lo;
      const int kv_end = ir.kv_end;
      const int j0 = ir.j0 + sg.it_lo;
      const int n_iter = sg.it_hi - sg.it_lo;
      int phys_next = (issuer && (j0 * BPT + bi) * 16 < kv_end) ? block_id(j0 * BPT + bi) : 0;
      for (int jj = 0; jj < n_iter && ok; ++jj, ++git) {
        const int j = j0 + jj;
        const int phys = phys_next;
        const int key0 = j * KT;
        const int lb = (j + 1) * BPT + bi;  // prefetch the next tile's block id
        phys_next = (issuer && lb * 16 < kv_end) ? block_id(lb) : 0;
        const int nblk = min(BPT, (kv_end - key0 + 15) / 16);
        // blocks of the item's first tile entirely before its first key are
        // not read (under local attention their pages may be gone)
        const int bskip = jj == 0 ? max(0, (kv_lo >> 4) - j * BPT) : 0;
        const int row = (phys * a.num_kv_heads + sg.kvh) * 16;
#pragma unroll 1
        for (int part = 0; part < 2; ++part) {
          if (part == 1 && jj == 0) {
            if (k > 0 && !mbar_wait(&bar[Q_EMPTY], (k - 1) & 1, a.wait_ns)) {
              ok = false;
              break;
            }
            // ---- the segment's Q tiles: a tile whose 128 / g queries all
            // belong to the chunk comes by TMA (16-bit caches, g dividing
            // 128); the others are staged by this warp (rows past the chunk
            // zeroed; with an 8-bit cache the bf16 queries become fp16)
            const int qs = ir.qs, qt0 = ir.qt0, nq = ir.nq;
            uint32_t qtma_tiles = 0;
            if (!C::KV8 && a.qtma) {
#pragma unroll
              for (int t = 0; t < NQT; ++t)
                if ((t + 1) * (MT / g) <= nq) qtma_tiles |= 1u << t;
            }
            if (qtma_tiles != (1u << NQT) - 1) {
              constexpr int CHUNKS = D / 8;  // 16-byte chunks per row
              float qmax = 0.f;
              for (int i = lane; i < MROWS * CHUNKS; i += 32) {
                const int R = i / CHUNKS;
                if (qtma_tiles >> (R / MT) & 1) continue;
                const int ch = i - R * CHUNKS;
                const int qi = R / g;
                const bool okr = R < rows_used && qi < nq;
                const uint16_t *src = a.q;
                if (okr)
                  src = a.q + (static_cast<int64_t>(qs + qt0 + qi) * a.num_q_heads + sg.kvh * g + (R - qi * g)) * D +
                        ch * 8;
                const int r = R & (MT - 1);
                uint8_t *dst =
                    smem + C::OFF_Q + (R / MT) * C::QB + (ch >> 3) * C::QHALF + r * 128 + (((ch & 7) ^ (r & 7)) << 4);
                if constexpr (C::KV8) {
                  uint4 y = make_uint4(0, 0, 0, 0);
                  if (okr) {
                    const uint4 x = __ldg(reinterpret_cast<const uint4 *>(src));
                    const uint32_t w[4] = {x.x, x.y, x.z, x.w};
                    uint32_t o[4];
#pragma unroll
                    for (int e = 0; e < 4; ++e) {
                      const float f0 = bf16lo(w[e]), f1 = bf16hi(w[e]);
                      qmax = fmaxf(qmax, fmaxf(fabsf(f0), fabsf(f1)));
                      o[e] = pack_f16x2(f0, f1);
                    }
                    y = make_uint4(o[0], o[1], o[2], o[3]);
                  }
                  *reinterpret_cast<uint4 *>(dst) = y;
                } else {
                  cp_async16(dst, src, okr);
                }
              }
              if (C::KV8 && qmax >= 65536.f && qmax <= FLT_MAX) report_error(a.err, a.ws_err, kErrFp16Range);
              cp_async_commit();
              cp_async_wait<0>();
              fence_proxy_async_smem();
              __syncwarp();
            }
            if (lane == 0) {
              if (qtma_tiles != 0) {
                mbar_arrive_expect_tx(&bar[Q_FULL], __popc(qtma_tiles) * C::QB);
#pragma unroll
                for (int t = 0; t < NQT; ++t)
                  if (qtma_tiles >> t & 1)
#pragma unroll
                    for (int q2 = 0; q2 < C::HALVES; ++q2)
                      tma_load_3d(smem + C::OFF_Q + t * C::QB + q2 * C::QHALF, &a.qmap, q2 * 64, sg.kvh * g,
                                  qs + qt0 + t * (MT / g), &bar[Q_FULL], pol);
                *s_last_q = k;
              } else {
                mbar_arrive(&bar[Q_FULL]);
              }
            }
            __syncwarp();
          }
          // K of iteration git (its slot frees once the QKs of git - NSK
          // completed), then V (once the PVs of git - NSV completed)
          const int st = part ? git % NSV : git % NSK;
          const uint32_t ph = part ? (git / NSV) & 1 : (git / NSK) & 1;
          const int full = (part ? V_FULL : K_FULL) + st;
          if (!mbar_wait(&bar[(part ? V_EMPTY : K_EMPTY) + st], ph ^ 1, a.wait_ns)) {
            ok = false;
            break;
          }
          if (!C::P16 && part == 1 && bskip > 0) {
            // V rows of the skipped blocks: zero (0 * NaN would not vanish in
            // the PV), before the copies of the other blocks start
            for (int i = lane; i < bskip * 16 * C::HALVES * 8; i += 32) {
              const int rr = i / (C::HALVES * 8);
              const int rem = i % (C::HALVES * 8);
              *reinterpret_cast<uint4 *>(smem + C::OFF_V + st * C::KVB + (rem >> 3) * C::KVHALF + rr * 128 +
                                         (rem & 7) * 16) = make_uint4(0, 0, 0, 0);
            }
            fence_proxy_async_smem();
          }
          if (lane == 0) mbar_arrive_expect_tx(&bar[full], (nblk - bskip) * C::BLOCK_BYTES);
          __syncwarp();
          if (issuer && bi < nblk && bi >= bskip) {
            uint8_t *slot = smem + (part ? C::OFF_V : C::OFF_K) + st * C::KVB;
            uint8_t *dst = C::KV8 ? slot + C::KVHALF + bi * 16 * D : slot + hh * C::KVHALF + bi * 16 * 128;
            tma_load_2d(dst, part ? &a.vmap : &a.kmap, hh * 64, row, &bar[full], pol);
          }
          if (lane == 0) *(part ? s_last_v : s_last_k) = git;
        }
      }
    }
    if (!ok && lane == 0) *s_abort = 1;
  } else if (warp == kMmaWarp) {
    // --------------------------------------------------------- MMA issuer
    // The grid kernel's order per KV iteration (PV_A, QK_A of the next
    // iteration, PV_B, QK_B of the next), where the next iteration may be
    // the next segment's first: its QKs wait for that segment's Q, and its
    // first PVs start O afresh.  A commit to Q_EMPTY follows each segment's
    // last QKs.
    if (lane == 0) {
      bool ok = true;
      auto qk = [&](int t, int gi) {  // S_t = Q_t K^T of iteration gi
        const uint32_t qbase = sbase + C::OFF_Q + t * C::QB;
        const uint32_t kbase = sbase + C::OFF_K + (gi % NSK) * C::KVB;
#pragma unroll
        for (int kk = 0; kk < D / 16; ++kk) {
          const uint64_t ad = umma_desc_sw128(qbase + (kk >> 2) * C::QHALF + (kk & 3) * 32, 16, 1024);
          const uint64_t bd = umma_desc_sw128(kbase + (kk >> 2) * C::KVHALF + (kk & 3) * 32, 16, 1024);
          umma_bf16_ss(tmem + t * KT, ad, bd, C::IDESC_QK, kk > 0 ? 1u : 0u);
        }
      };
      auto pv = [&](int t, int gi, bool acc) {  // O_t (+)= P_t V of iteration gi, P_t from TMEM
        const uint32_t vbase = sbase + C::OFF_V + (gi % NSV) * C::KVB;
        constexpr int NPART = C::P16 ? 1 : 2;
#pragma unroll
        for (int part = 0; part < NPART; ++part) {
#pragma unroll
          for (int kk = 0; kk < KT / 16; ++kk) {
            const uint64_t bd = umma_desc_sw128(vbase + kk * 2048, C::KVHALF, 1024);
            umma_bf16_ts(tmem + C::O_COL + t * D, tmem + t * KT + (kk >> 1) * 32 + part * 16 + (kk & 1) * 8, bd,
                         C::IDESC_PV, (acc || part > 0 || kk > 0) ? 1u : 0u);
          }
        }
      };
      constexpr int VB = C::P16 ? V_READY : V_FULL;
      constexpr int KB = C::KV8 ? K_READY : K_FULL;
      SkIter iter = it0;
      Seg cur, nxt;
      bool has_cur = iter.next(a, cur);
      bool has_nxt = has_cur && iter.next(a, nxt);
      if (has_cur) {
        // the first QKs need Q and K only; V of the first tile is waited
        // for behind them
        if (!mbar_wait(&bar[Q_FULL], 0, a.wait_ns) || !mbar_wait(&bar[KB], 0, a.wait_ns)) ok = false;
        if (ok) {
          tc_fence_after_sync();
          for (int t = 0; t < NQT; ++t) {
            qk(t, 0);
            umma_commit(&bar[S_FULL + t]);
          }
          if (cur.it_hi - cur.it_lo == 1) umma_commit(&bar[Q_EMPTY]);
          if (!mbar_wait(&bar[VB], 0, a.wait_ns)) ok = false;
        }
      }
      int git = 0;
      for (int k = 0; ok && has_cur; ++k) {
        const int n = cur.it_hi - cur.it_lo;
        for (int jj = 0; jj < n && ok; ++jj, ++git) {
          const bool has_next = jj + 1 < n || has_nxt;         // another iteration follows
          const bool next_first = jj + 1 == n && has_nxt;      // ... the next segment's first
          const bool next_last = next_first ? nxt.it_hi - nxt.it_lo == 1 : jj + 2 == n;  // ... its segment's last
          for (int t = 0; t < NQT; ++t) {
            if (!mbar_wait_hint(&bar[P_FULL + t], git & 1, a.wait_ns)) {
              ok = false;
              break;
            }
            tc_fence_after_sync();
            pv(t, git, jj > 0);
            if (t == NQT - 1) {
              umma_commit(&bar[V_EMPTY + git % NSV]);  // both tiles are done with V of iteration git
              if (has_next && !mbar_wait(&bar[VB + (git + 1) % NSV], ((git + 1) / NSV) & 1, a.wait_ns)) {
                ok = false;
                break;
              }
            }
            if (has_next) {
              if (t == 0) {
                if (!mbar_wait(&bar[KB + (git + 1) % NSK], ((git + 1) / NSK) & 1, a.wait_ns) ||
                    (next_first && !mbar_wait(&bar[Q_FULL], (k + 1) & 1, a.wait_ns))) {
                  ok = false;
                  break;
                }
              }
              tc_fence_after_sync();
              qk(t, git + 1);
              if (t == NQT - 1 && next_last) umma_commit(&bar[Q_EMPTY]);  // the segment's Q is free
            }
            // S_t of the next iteration is ready and PV_t(git) has completed
            // (after a segment's last iteration: its O_t is final)
            umma_commit(&bar[S_FULL + t]);
            if (t == 0) umma_commit(&bar[K_EMPTY + git % NSK]);  // both tiles are done with K of iteration git
          }
        }
        cur = nxt;
        has_cur = has_nxt;
        has_nxt = has_cur && iter.next(a, nxt);
      }
      if (!ok) *s_abort = 1;
    }
    __syncwarp();
  } else if (C::P16 && warp >= kConvWarp0 && warp < kConvWarp0 + 2) {
    // --------------------------------- K / V tile preparation (fp16 P)
    // as in the grid kernel, per KV iteration of every segment: V rows
    // outside the segment's keys zeroed, bf16 V converted to fp16, 8-bit K
    // and V widened to fp16
    const int ct = tid - kConvWarp0 * 32;
    bool ok = true;
    float vmax = 0.f;
    constexpr int UNITS = C::KVB / 16;
    constexpr int UROW = KT * 8;
    auto widen8 = [&](uint8_t *slot, int r_lo, int r_hi, bool zero_rows) {
      const uint8_t *land = slot + C::KVHALF;
      auto put = [&](int half, int r, int c4, const uint4 &x) {
        const bool keep = !zero_rows || (r >= r_lo && r < r_hi);
        const uint32_t w[4] = {x.x, x.y, x.z, x.w};
        uint32_t o[8];
#pragma unroll
        for (int e = 0; e < 4; ++e) {
          o[2 * e] = fp8x2_to_f16x2<KVT>(static_cast<uint16_t>(w[e] & 0xffffu));
          o[2 * e + 1] = fp8x2_to_f16x2<KVT>(static_cast<uint16_t>(w[e] >> 16));
        }
        uint8_t *row = slot + half * C::KVHALF + r * 128;
        const int k0 = 2 * c4, k1 = 2 * c4 + 1;
        *reinterpret_cast<uint4 *>(row + ((k0 ^ (r & 7)) << 4)) =
            keep ? make_uint4(o[0], o[1], o[2], o[3]) : make_uint4(0, 0, 0, 0);
        *reinterpret_cast<uint4 *>(row + ((k1 ^ (r & 7)) << 4)) =
            keep ? make_uint4(o[4], o[5], o[6], o[7]) : make_uint4(0, 0, 0, 0);
      };
#pragma unroll 2
      for (int u = ct; u < KT * 4; u += 64) {
        const int r = u >> 2, c = u & 3;
        put(0, r, c, *reinterpret_cast<const uint4 *>(land + r * 128 + ((c ^ (r & 7)) << 4)));
      }
      constexpr int PER = KT * 4 / 64;
      uint4 x[PER];
#pragma unroll
      for (int k = 0; k < PER; ++k) {
        const int u = ct + 64 * k, r = u >> 2, c = 4 + (u & 3);
        x[k] = *reinterpret_cast<const uint4 *>(land + r * 128 + ((c ^ (r & 7)) << 4));
      }
      named_bar_sync(2, 64);  // every read of the landed bytes is done
#pragma unroll
      for (int k = 0; k < PER; ++k) {
        const int u = ct + 64 * k;
        put(1, u >> 2, u & 3, x[k]);
      }
    };
    SkIter iter = it0;
    Seg sg;
    int git = 0;
    while (ok && iter.next(a, sg)) {
      ItemRange ir;
      item_range(a, sg.s, 0, sg.qtile, sg.gx, false, ir);
      const int j0 = ir.j0 + sg.it_lo;
      const int n_iter = sg.it_hi - sg.it_lo;
      for (int jj = 0; jj < n_iter; ++jj, ++git) {
        const int key0 = (j0 + jj) * KT;
        const int r_lo = max(ir.kv_lo - key0, 0);
        const int r_hi = min(ir.kv_end - key0, KT);
        if constexpr (C::KV8) {
          const int stk = git % NSK;
          if (!named_bar_and(2, 64, mbar_wait(&bar[K_FULL + stk], (git / NSK) & 1, a.wait_ns))) {
            ok = false;
            break;
          }
          widen8(smem + C::OFF_K + stk * C::KVB, r_lo, r_hi, false);
          fence_proxy_async_smem();
          __syncwarp();
          if (lane == 0) mbar_arrive(&bar[K_READY + stk]);
        }
        const int st = git % NSV;
        if (!named_bar_and(2, 64, mbar_wait(&bar[V_FULL + st], (git / NSV) & 1, a.wait_ns))) {
          ok = false;
          break;
        }
        uint4 *vt = reinterpret_cast<uint4 *>(smem + C::OFF_V + st * C::KVB);
        if constexpr (C::KV8) {
          widen8(smem + C::OFF_V + st * C::KVB, r_lo, r_hi, true);
        } else if constexpr (C::CONVERT) {
          constexpr int ILP = 8;
          static_assert(UNITS % (64 * ILP) == 0, "whole steps");
#pragma unroll 1
          for (int u0 = ct; u0 < UNITS; u0 += 64 * ILP) {
            uint4 x[ILP];
#pragma unroll
            for (int k = 0; k < ILP; ++k) x[k] = vt[u0 + 64 * k];
#pragma unroll
            for (int k = 0; k < ILP; ++k) {
              const int row = ((u0 + 64 * k) % UROW) >> 3;
              const uint32_t w[4] = {x[k].x, x[k].y, x[k].z, x[k].w};
              uint32_t y[4];
              float um = 0.f;
#pragma unroll
              for (int e = 0; e < 4; ++e) {
                const float f0 = bf16lo(w[e]), f1 = bf16hi(w[e]);
                um = fmaxf(um, fmaxf(fabsf(f0), fabsf(f1)));
                y[e] = pack_f16x2(f0, f1);
              }
              const bool keep = row >= r_lo && row < r_hi;
              if (keep) vmax = fmaxf(vmax, um);
              vt[u0 + 64 * k] = keep ? make_uint4(y[0], y[1], y[2], y[3]) : make_uint4(0, 0, 0, 0);
            }
          }
        } else if (r_lo > 0 || r_hi < KT) {
          for (int u = ct; u < UNITS; u += 64) {
            const int row = (u % UROW) >> 3;
            if (row < r_lo || row >= r_hi) vt[u] = make_uint4(0, 0, 0, 0);
          }
        }
        fence_proxy_async_smem();
        __syncwarp();
        if (lane == 0) mbar_arrive(&bar[V_READY + st]);
      }
    }
    if (C::CONVERT && vmax >= 65536.f && vmax <= FLT_MAX) report_error(a.err, a.ws_err, kErrFp16Range);
    if (!ok && lane == 0) *s_abort = 1;
  } else if (warp >= kSoftmaxWarp0) {
    // ------------------------------------- softmax, two threads per row
    // As in the grid kernel (see there), per segment; then the segment's
    // output: a whole item straight to out (the last segment's full tiles
    // through shared memory and TMA stores), a piece to its slot and, if it
    // completes the item, the merge of all its pieces.
    const int h = (warp - kSoftmaxWarp0) >> 2;
    const int r = ((warp & 3) << 5) | lane;
    const uint32_t trow = tmem + (static_cast<uint32_t>((warp & 3) * 32) << 16);
    float *xch = reinterpret_cast<float *>(smem + C::OFF_X);
    const int pair_bar = 3 + (warp & 3);
    SkIter iter = it0;
    Seg sg;
    int git = 0;
    bool ok = true;
    bool stored = false;  // TMA stores of output tiles issued by this thread
    while (ok && iter.next(a, sg)) {
      ItemRange ir;
      item_range(a, sg.s, 0, sg.qtile, sg.gx, false, ir);
      const int kvh = sg.kvh;
      const int qs = ir.qs, qt0 = ir.qt0, nq = ir.nq;
      const int j0 = ir.j0 + sg.it_lo;
      const int n_iter = sg.it_hi - sg.it_lo;
      const float qscale = a.k_scales ? a.qscale0 * __ldg(a.k_scales + kvh) : a.qscale;
      const float vscale = a.v_scales ? __ldg(a.v_scales + kvh) : a.vscale;
      float m_ref[NQT], l[NQT];
      int pos[NQT], first[NQT];
#pragma unroll
      for (int t = 0; t < NQT; ++t) {
        const int R = t * MT + r;
        const int qi = R / g;
        const bool rv = R < rows_used && qi < nq;
        pos[t] = rv ? ir.base_pos + qi : -1;  // keys <= pos are visible
        first[t] = local_first_key(pos[t], a.window, a.chunk);  // ... and keys >= first
        m_ref[t] = -INFINITY;
        l[t] = 0.f;
      }
      for (int jj = 0; jj < n_iter && ok; ++jj, ++git) {
        const int key0 = (j0 + jj) * KT;
#pragma unroll
        for (int t = 0; t < NQT; ++t) {
          bool got = mbar_wait_hint(&bar[S_FULL + t], git & 1, a.wait_ns);
          tc_fence_after_sync();
          const uint32_t s_col = t * KT;
          const uint32_t o_col = C::O_COL + t * D;
          if (!C::P16 && t == 0 && h == 0 && jj == n_iter - 1 && ir.kv_end - key0 < KT && got) {
            // pair mode: V rows past the last needed key are zeroed, after
            // this tile's V copies landed
            got = mbar_wait(&bar[V_FULL + git % NSV], (git / NSV) & 1, a.wait_ns);
            const int kval = ir.kv_end - key0;
            for (int i = r; got && i < (KT - kval) * C::HALVES * 8; i += MT) {
              const int row = kval + i / (C::HALVES * 8);
              const int rem = i % (C::HALVES * 8);
              *reinterpret_cast<uint4 *>(smem + C::OFF_V + (git % NSV) * C::KVB + (rem >> 3) * C::KVHALF +
                                         row * 128 + (rem & 7) * 16) = make_uint4(0, 0, 0, 0);
            }
            fence_proxy_async_smem();
          }
          if (!named_bar_and(pair_bar, 64, got)) {
            ok = false;
            break;
          }
          uint32_t sc[2][32];
          tmem_ld32_async(trow + s_col + (2 * h) * 32, sc[0]);
          tmem_ld32_async(trow + s_col + (2 * h + 1) * 32, sc[1]);
          tmem_wait_ld(sc[0]);
          tmem_wait_ld(sc[1]);
          const int kh = key0 + h * 64;
          float mx = -INFINITY;
#pragma unroll
          for (int c = 0; c < 2; ++c) {
            const int kc = kh + c * 32;
            if (!(kc + 31 <= pos[t] && kc >= first[t])) {
#pragma unroll
              for (int i = 0; i < 32; ++i)
                if (kc + i > pos[t] || kc + i < first[t]) sc[c][i] = __float_as_uint(-INFINITY);
            }
            float m[11];
#pragma unroll
            for (int i = 0; i < 10; ++i)
              m[i] = fmax3(__uint_as_float(sc[c][3 * i]), __uint_as_float(sc[c][3 * i + 1]),
                           __uint_as_float(sc[c][3 * i + 2]));
            m[10] = fmaxf(__uint_as_float(sc[c][30]), __uint_as_float(sc[c][31]));
            mx = fmax3(mx, fmax3(fmax3(m[0], m[1], m[2]), fmax3(m[3], m[4], m[5]), fmax3(m[6], m[7], m[8])),
                       fmaxf(m[9], m[10]));
          }
          xch[h * MT + r] = mx;
          named_bar_sync(pair_bar, 64);
          mx = fmaxf(mx, xch[(h ^ 1) * MT + r]) * qscale;
          const float m_new = fmaxf(m_ref[t], mx);
          const bool raise =
              m_new > m_ref[t] + kRescaleThreshold || (m_ref[t] == -INFINITY && m_new != -INFINITY);
          if (__any_sync(0xffffffffu, raise && m_ref[t] != -INFINITY)) {
            const float corr = (raise && m_ref[t] != -INFINITY) ? exp2f(m_ref[t] - m_new) : 1.f;
            if (raise) l[t] *= corr;
            if (jj > 0) {
#pragma unroll 1
              for (int c0 = h * (D / 2); c0 < (h + 1) * (D / 2); c0 += 32) {
                float o[32];
                tmem_ld32(trow + o_col + c0, o);
#pragma unroll
                for (int i = 0; i < 32; ++i) o[i] *= corr;
                tmem_st32(trow + o_col + c0, o);
              }
            }
          }
          if (raise) m_ref[t] = m_new;
          const float nref = (m_ref[t] == -INFINITY) ? 0.f : -m_ref[t];
          const uint64_t qs2 = f2_pack(qscale, qscale), nr2 = f2_pack(nref, nref);
          uint64_t lsum[2] = {0, 0};
#pragma unroll
          for (int c = 0; c < 2; ++c) {
            uint32_t hi[16], lo[16];
#pragma unroll
            for (int e = 0; e < 16; ++e) {
              const float2 x = f2_unpack(
                  f2_fma(f2_pack(__uint_as_float(sc[c][2 * e]), __uint_as_float(sc[c][2 * e + 1])), qs2, nr2));
              const float p0 = ex2_approx(x.x);
              const float p1 = ex2_approx(x.y);
              const uint64_t pp = f2_pack(p0, p1);
              lsum[e & 1] = f2_add(lsum[e & 1], pp);
              if constexpr (C::P16) {
                hi[e] = pack_f16x2(p0, p1);
              } else {
                hi[e] = pack16x2<KVT>(p0, p1);
                const float2 d = f2_unpack(f2_sub(pp, f2_pack(lo16<KVT>(hi[e]), hi16<KVT>(hi[e]))));
                lo[e] = pack16x2<KVT>(d.x, d.y);
              }
            }
            tmem_st16_async(trow + s_col + (2 * h + c) * 32, hi);
            if constexpr (!C::P16) tmem_st16_async(trow + s_col + (2 * h + c) * 32 + 16, lo);
          }
          {
            const float2 l2 = f2_unpack(f2_add(lsum[0], lsum[1]));
            l[t] += l2.x + l2.y;
          }
          tmem_wait_st();
          tc_fence_before_sync();
          __syncwarp();
          if (lane == 0) mbar_arrive(&bar[P_FULL + t]);
        }
      }
      // ---- the segment's output.  The row sums of both halves (both warps
      // of a pair take part, even after a timeout, so that the pair's named
      // barriers stay matched)
      float lt[NQT];
#pragma unroll
      for (int t = 0; t < NQT; ++t) {
        named_bar_sync(pair_bar, 64);
        xch[h * MT + r] = l[t];
        named_bar_sync(pair_bar, 64);
        lt[t] = l[t] + xch[(h ^ 1) * MT + r];
      }
      const bool last_seg = !iter.more();
      if (!sg.piece) {
#pragma unroll
        for (int t = 0; t < NQT; ++t) {
          // the commit after this segment's last PV_t (git: one past its last iteration)
          if (ok && !mbar_wait(&bar[S_FULL + t], git & 1, a.wait_ns)) ok = false;
          if (!ok) break;
          tc_fence_after_sync();
          const int R = t * MT + r;
          const int qi = R / g;
          const bool rv = R < rows_used && qi < nq;
          const uint32_t o_col = C::O_COL + t * D;
          const float inv = lt[t] > 0.f ? vscale / lt[t] : 0.f;
          const int64_t orow_i = static_cast<int64_t>(qs + qt0 + qi) * a.num_q_heads + kvh * g + (R - qi * g);
          if (last_seg && a.otma && (t + 1) * (MT / g) <= nq) {
            // the CTA's last segment, a full tile: through shared memory (the
            // K ring and beyond, free once the last products completed) and
            // out by TMA stores, as in the grid kernel
            uint8_t *stage = smem + C::OFF_K + t * (D / 32) * 16384;
#pragma unroll 1
            for (int c0 = h * (D / 2); c0 < (h + 1) * (D / 2); c0 += 32) {
              float o[32];
              tmem_ld32(trow + o_col + c0, o);
              uint8_t *rowp = stage + (c0 / 32) * 16384 + r * 128;
#pragma unroll
              for (int k = 0; k < 8; ++k)
                *reinterpret_cast<float4 *>(rowp + ((k ^ (r & 7)) << 4)) =
                    make_float4(o[4 * k] * inv, o[4 * k + 1] * inv, o[4 * k + 2] * inv, o[4 * k + 3] * inv);
            }
            fence_proxy_async_smem();
            named_bar_sync(7 + h, 128);
            if ((warp & 3) == 0 && lane == 0) {
              for (int c0 = h * (D / 2); c0 < (h + 1) * (D / 2); c0 += 32)
                tma_store_3d(&a.omap, stage + (c0 / 32) * 16384, c0, kvh * g, qs + qt0 + t * (MT / g));
              bulk_commit_group();
              stored = true;
            }
          } else {
#pragma unroll 1
            for (int c0 = h * (D / 2); c0 < (h + 1) * (D / 2); c0 += 32) {
              float o[32];
              tmem_ld32(trow + o_col + c0, o);
              if (rv) {
                float *orow = a.out + orow_i * D;
#pragma unroll
                for (int i = 0; i < 32; i += 4)
                  *reinterpret_cast<float4 *>(orow + c0 + i) =
                      make_float4(o[i] * inv, o[i + 1] * inv, o[i + 2] * inv, o[i + 3] * inv);
              }
            }
          }
          if (rv && h == 0 && a.lse) a.lse[orow_i] = (m_ref[t] + log2f(lt[t])) * kLn2;
        }
      } else {
        // a piece: its normalised O ([Q tile][D / 4][MT] float4, a warp's
        // rows side by side) and its log-sum-exp (log2 units) to its slot
        float4 *po = reinterpret_cast<float4 *>(a.part_o) + static_cast<int64_t>(sg.slot) * NQT * (D / 4) * MT;
        float *pl = a.part_lse + static_cast<int64_t>(sg.slot) * MROWS;
#pragma unroll
        for (int t = 0; t < NQT; ++t) {
          if (ok && !mbar_wait(&bar[S_FULL + t], git & 1, a.wait_ns)) ok = false;
          if (!ok) break;
          tc_fence_after_sync();
          const int R = t * MT + r;
          const int qi = R / g;
          const bool rv = R < rows_used && qi < nq;
          const float inv = lt[t] > 0.f ? 1.f / lt[t] : 0.f;
#pragma unroll 1
          for (int c0 = h * (D / 2); c0 < (h + 1) * (D / 2); c0 += 32) {
            float o[32];
            tmem_ld32(trow + C::O_COL + t * D + c0, o);
            if (rv) {
#pragma unroll
              for (int k = 0; k < 8; ++k)
                po[(t * (D / 4) + c0 / 4 + k) * MT + r] = make_float4(__fmul_rn(o[4 * k], inv), __fmul_rn(o[4 * k + 1], inv),
                                                           __fmul_rn(o[4 * k + 2], inv), __fmul_rn(o[4 * k + 3], inv));
            }
          }
          if (rv && h == 0) pl[R] = lt[t] > 0.f ? m_ref[t] + log2f(lt[t]) : -INFINITY;
        }
        // count the piece once all 256 softmax threads stored theirs and went
        // on (after a timeout the item stays unmerged; the timeout is reported)
        __threadfence();
        if (named_bar_and(9, 256, ok)) {
          if (tid == kSoftmaxWarp0 * 32) {
            const int prev = atom_add_acq_rel_gpu(a.part_count + sg.item, 1);
            if (prev == sg.c_hi - sg.c_lo) {
              // the item's last piece: this CTA merges them, once its
              // pipeline has drained (sk_run_merges)
              st_relaxed_gpu(a.part_count + sg.item, 0);  // ready for the next launch
              int *nm = reinterpret_cast<int *>(smem + C::OFF_M);
              SkMerge *ml = reinterpret_cast<SkMerge *>(smem + C::OFF_M + 16);
              if (*nm < kMaxMerges) ml[(*nm)++] = SkMerge{sg.item_start, sg.c_lo, sg.c_hi, qs, qt0, nq, kvh, vscale};
            }
          }
        } else {
          ok = false;
        }
      }
      // every softmax thread goes on to the next segment, or none does
      ok = named_bar_and(9, 256, ok);
    }
    // the stores' shared-memory sources are read before the CTA exits
    if (stored) bulk_wait_group_read0();
    if (!ok && lane == 0) *s_abort = 1;
  }

  // ---- teardown: after an abort the copies still in flight land first;
  // every product completes before the tensor memory is freed
  tc_fence_before_sync();
  __syncthreads();
  if (*s_abort) {
    if (tid == 0) report_error(a.err, a.ws_err, kErrWaitTimeout);
    if (warp == kProducerWarp && lane == 0) {
      if (*s_last_q >= 0) mbar_wait(&bar[Q_FULL], *s_last_q & 1, a.wait_ns);
      for (int t = max(0, *s_last_k - NSK + 1); t <= *s_last_k; ++t)
        mbar_wait(&bar[K_FULL + t % NSK], (t / NSK) & 1, a.wait_ns);
      for (int t = max(0, *s_last_v - NSV + 1); t <= *s_last_v; ++t)
        mbar_wait(&bar[V_FULL + t % NSV], (t / NSV) & 1, a.wait_ns);
    }
  }
  if (warp == kMmaWarp && lane == 0) {
    // a commit after everything this thread issued: its arrival follows the
    // completion of every product
    uint64_t *drain = &bar[P_FULL];
    mbar_init(drain, 1);
    fence_mbar_init();
    umma_commit(drain);
    mbar_wait(drain, 0, a.wait_ns);
  }
  tc_fence_before_sync();
  __syncthreads();
  // the merges this CTA owes (the pieces of other CTAs were complete when it
  // counted its own: their stores precede their counts)
  const int nmerge = *reinterpret_cast<volatile int *>(smem + C::OFF_M);
  if (nmerge > 0 && !*s_abort) {
    __threadfence();
    sk_run_merges<D, KVT, PVM>(a, smem, it0.U, it0.G, nmerge);
  }
}

// The balanced launch: one CTA per SM (see the file comment).  Each CTA
// computes the prefix sums of the pairs' iterations in shared memory (the K
// ring, before any copy), finds its range's first and last items, then runs
// its segments.  Chunk mode only.
template <int D, int KVT, int PVM>
__global__ void __launch_bounds__(NTHREADS, 1) prefill_sk_kernel(const __grid_constant__ Args a) {
  using C = Cfg<D, KVT, PVM>;
  asm volatile("griddepcontrol.wait;" ::: "memory");
  extern __shared__ uint8_t smem_raw[];
  uint8_t *smem = align1024(smem_raw);
  uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(smem + C::OFF_BAR + NBAR * 8);
  const int tid = threadIdx.x;
  const int warp = tid >> 5;
  const int lane = tid & 31;
  if (warp == kMmaWarp) tmem_alloc(tmem_slot, C::TMEM_COLS);

  // ---- prefix sums ps[p] of the pairs' iterations (ps[P]: all of them)
  const int P = a.num_seqs * a.gx;
  int *ps = reinterpret_cast<int *>(smem + C::OFF_K);   // [P + 1]
  int *wsum = reinterpret_cast<int *>(smem + C::OFF_X);  // [NTHREADS / 32]
  const int per = (P + NTHREADS - 1) / NTHREADS;
  const int lo = min(P, tid * per), hi = min(P, lo + per);
  int run = 0;
  for (int p = lo; p < hi; ++p) {
    const int n = pair_iters(a, p);
    ps[p] = n;
    run += n;
  }
  int incl = run;  // inclusive scan of the threads' sums: in the warp ...
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const int v = __shfl_up_sync(0xffffffffu, incl, o);
    if (lane >= o) incl += v;
  }
  if (lane == 31) wsum[warp] = incl;
  __syncthreads();
  if (warp == 0) {  // ... then over the warps
    int w = lane < NTHREADS / 32 ? wsum[lane] : 0;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const int v = __shfl_up_sync(0xffffffffu, w, o);
      if (lane >= o) w += v;
    }
    if (lane < NTHREADS / 32) wsum[lane] = w;
  }
  __syncthreads();
  int base = (warp > 0 ? wsum[warp - 1] : 0) + incl - run;
  for (int p = lo; p < hi; ++p) {
    const int n = ps[p];
    ps[p] = base;
    base += n;
  }
  if (tid == NTHREADS - 1) ps[P] = base;
  __syncthreads();

  // ---- this CTA's units [u0, u1): at least 4 per CTA (a small launch is
  // shared by fewer CTAs; the others only free their tensor memory)
  SkIter itr;
  itr.H = a.num_kv_heads;
  itr.P = P;
  itr.T = ps[P];
  itr.U = itr.T * itr.H;
  itr.G = max(1, min(static_cast<int>(gridDim.x), itr.U / 4));
  itr.me = blockIdx.x;
  const int u0 = itr.me < itr.G ? sk_first_unit(itr.me, itr.U, itr.G) : itr.U;
  const int u1 = itr.me < itr.G ? sk_first_unit(itr.me + 1, itr.U, itr.G) : itr.U;
  // the item holding unit u: kv head u / T, then the largest pair p with
  // ps[p] <= u % T (pairs without iterations share their successor's
  // prefix, so it has iterations)
  auto locate = [&](int u, int &p, int &kv) {
    kv = u / itr.T;
    const int rem = u - kv * itr.T;
    int l = 0, r = P - 1;
    while (l < r) {
      const int m = (l + r + 1) >> 1;
      if (ps[m] <= rem) l = m;
      else r = m - 1;
    }
    p = l;
  };
  itr.u = itr.ub = itr.u1 = u1;
  itr.z_first = 0;
  if (u0 < u1) {
    locate(u0, itr.p, itr.kvh);
    itr.np = ps[itr.p + 1] - ps[itr.p];
    itr.base = itr.kvh * itr.T + ps[itr.p];
    itr.it = u0 - itr.base;
    itr.u = u0;
    locate(u1 - 1, itr.pz, itr.kvz);
    itr.nz = ps[itr.pz + 1] - ps[itr.pz];
    itr.zs = itr.kvz * itr.T + ps[itr.pz];
    itr.z_first = itr.zs > u0 && itr.zs + itr.nz > u1;
    itr.ub = itr.z_first ? itr.zs : u1;
  }
  tc_fence_before_sync();
  __syncthreads();  // every read of the prefix sums is done: the K ring is free
  tc_fence_after_sync();
  const uint32_t tmem = *tmem_slot;
  if (u0 < u1) prefill_run<D, KVT, PVM>(a, smem, tmem, itr);
  tc_fence_before_sync();
  __syncthreads();
  if (warp == kMmaWarp) {
    tc_fence_after_sync();
    tmem_dealloc(tmem, C::TMEM_COLS);
  }
}

}  // namespace pftc
}  // namespace pa
