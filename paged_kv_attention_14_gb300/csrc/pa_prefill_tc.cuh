// pa_prefill_tc.cuh -- causal chunked-prefill attention on the 5th-generation
// tensor cores (tcgen05.mma, accumulators in tensor memory): bf16, fp16 or
// 8-bit (E4M3, E5M2) KV.
//
// What it computes is the same as pa_prefill.cu: sequence s brings q_len
// new queries (a "chunked prefill" chunk, vllm.cpp implementation notes,
// Engine core bullet); query i sits at position context_lens[s] - q_len + i
// and attends keys [0, position] through the block table, reading blocks
// that may be shared with other sequences ("Zero-Copy Cache Hits" of "1.
// Technical Mechanics of the Radix Cache", Building and Deploying vllm.cpp).
//
// How (GB300 design):
//  * One CTA takes 256 (query, head) rows: 256 / g consecutive queries of
//    one sequence times the g query heads of one kv head, so every K/V tile
//    feeds the whole GQA group.  The rows form two 128-row Q tiles (A, B)
//    that ping-pong: while one tile's softmax runs, the tensor cores work on
//    the other tile.  A Q tile whose queries all belong to the chunk comes
//    by TMA (16-bit caches, g dividing 128), issued together with the first
//    K/V copies; other tiles are staged by the threads.  K/V are walked in
//    128-key tiles gathered block by block through the block table by TMA
//    (128-byte-swizzled boxes of 16 rows) into a 3-stage K ring and a
//    2-stage V ring shared by both Q tiles.  A K slot is released as soon
//    as the QKs that read it complete, a V slot after its PVs.
//  * Warp 0 (one thread) issues the MMAs.  S_t = Q_t K^T (M 128, N 128 keys,
//    K 16 x head_dim/16; both operands in shared memory) lands in tile t's
//    128 TMEM columns.  The softmax overwrites those columns with P_t: one
//    fp16 value per key (kPvF16, the default), or a hi + lo pair of the
//    cache's 16-bit type in pair mode (P = hi + lo to ~2^-17 relative with
//    bf16).  O_t += P_t V (M 128, N head_dim, K 16 x 8, twice in pair mode)
//    takes P_t straight from tensor memory as the A operand and V MN-major
//    from shared memory.  Order per KV tile j: PV_A(j), QK_A(j+1), PV_B(j),
//    QK_B(j+1); one commit after each QK tells tile t's softmax that its
//    next scores are ready AND that its previous PV finished (so O_t may be
//    rescaled and S_t overwritten).  M 128 MMAs with N <= 128 cost the same
//    per instruction (measured on GB300: ~84 cycles with both operands in
//    shared memory, ~78 with A in tensor memory, 128 at N 256), hence the
//    128-key tile.
//  * With fp16 P, warps 2-3 prepare each landed V tile: a bf16 tile is
//    converted to fp16 in place (both MMA operands are then fp16), and rows
//    outside the keys the CTA needs are zeroed (0 * NaN would not vanish).
//    8-bit K and V tiles are widened to fp16 in place, and the queries are
//    then staged in fp16.
//  * Warps 4-11 do the online softmax, two threads per row: warps 4-7 take
//    keys 0-63 and warps 8-11 keys 64-127 of every tile, for tile A and then
//    tile B.  Per tile: the scores from TMEM, causal and local masks, the
//    half-row max (a tree of three-input maxima) exchanged with the partner
//    thread through shared memory, exp2 of the scaled scores, the row sum
//    and P, with packed fp32x2 arithmetic.  The running max is only raised
//    (and O rescaled in TMEM) when it grows by more than 2^8, so that path
//    is rare.
//  * Warp 1 issues the TMA copies and prefetches block-table entries one
//    tile ahead.
//  * Every wait is bounded; on a timeout the kernel records an error bit,
//    lets its own MMAs and copies drain and frees its TMEM before returning.
#pragma once

#include <cuda.h>
#include <float.h>
#include <string.h>

#include "pa_device.cuh"
#include "pa_host_cache.h"
#include "pa_internal.h"

namespace pa {
namespace pftc {

constexpr float kLog2e = 1.4426950408889634f;
constexpr float kLn2 = 0.6931471805599453f;
constexpr int KT = 128;        // keys per KV tile (N of the QK MMA)
constexpr int BPT = KT / 16;   // cache blocks per KV tile
constexpr int MT = 128;        // rows of one Q tile (one TMEM lane per row)
constexpr int NQT = 2;         // Q tiles per CTA (their softmaxes alternate with their MMAs)
constexpr int MROWS = MT * NQT;
// Warp roles.  The MMA issuer and the TMA producer take the lowest warp
// numbers: they must be scheduled promptly on sub-partitions shared with
// busy softmax warps, and the warp schedulers favour older warps.  Softmax
// warp w may only touch TMEM lanes 32 (w % 4) .. 32 (w % 4) + 31, so each
// half of the keys' warpgroup starts at a multiple of four.
constexpr int NTHREADS = 384;  // warp 0 MMA issuer, 1 TMA producer, 2-3 K / V preparation, 4-11 softmax
constexpr int kMmaWarp = 0;
constexpr int kProducerWarp = 1;
constexpr int kSoftmaxWarp0 = 4;
constexpr int kConvWarp0 = 2;  // fp16 P: warps 2-3 prepare the V tiles
constexpr int NSK = 3;         // stages of the K ring
constexpr int NSV = 2;         // stages of the V ring
constexpr float kRescaleThreshold = 8.f;  // log2 units

struct Args {
  CUtensorMap kmap;  // cache as [rows = blocks * kv heads * 16][D], box {64, 16}
  CUtensorMap vmap;
  // queries as [tokens][q heads][D] of 16-bit values, box {64, g, 128 / g}:
  // one box is one 128-byte column half of a Q tile (its 128 / g queries
  // times the g heads of one kv head).  Used when qtma is set.
  CUtensorMap qmap;
  int qtma;          // the full Q tiles come by TMA (16-bit caches, g divides 128)
  // the output as [tokens][q heads][D] fp32, box {32, g, 128 / g}: one box
  // is 32 columns of an output tile, in the order of its rows.  Used when
  // otma is set (chunk mode, g divides 128).
  CUtensorMap omap;
  int otma;
  float *out;
  float *lse;
  const uint16_t *q;
  const int32_t *query_start_loc;
  const int32_t *block_tables;
  const int32_t *context_lens;
  int max_blocks_per_seq;
  int num_kv_heads;
  int num_q_heads;
  int g;
  int qt;  // queries per CTA (256 / g)
  float qscale;     // scale * k_scale * log2(e)
  float qscale0;    // scale * log2(e) (8-bit caches with per-head scales)
  float vscale;     // v_scale (8-bit caches; 1 otherwise)
  const float *k_scales;  // per-kv-head scales of an 8-bit cache, or NULL
  const float *v_scales;
  int window;  // local attention (see pa_kv_desc), 0: none
  int chunk;
  int prefix_mode;  // 1: every query after all L keys, no causal mask (shared prefix)
  int num_splits;   // prefix mode: key splits per sequence (grid.z = sequences x splits)
  int split_len;    // prefix mode: keys per split (a multiple of KT)
  int out_slots;    // prefix mode: output slots per (row, head); split i writes slot i
  int32_t *err;     // the caller's error word (pa_kv_desc.error_word), or NULL
  unsigned long long wait_ns;  // limit of every bounded wait
  int checked;      // range-check block ids and lengths (pa_kv_desc.check_indices)
  int stall;        // test hook: the producer issues nothing, so the waits run out
  int num_blocks;   // blocks of the cache (checked mode)
  // balanced launch (prefill_sk_kernel): items are (pair p, kv head), pair p
  // = (sequence p / gx, query tile gx - 1 - p % gx), and their KV iterations
  // are dealt out evenly over the CTAs.  An item cut between CTAs leaves one
  // piece per CTA in a slot (two slots per CTA: its first and its last item)
  int num_seqs;
  int gx;               // query tiles per sequence
  float *part_o;        // [2 G][NQT][D / 4][MT] float4: normalised O of a piece
  float *part_lse;      // [2 G][MROWS]: its log-sum-exp, log2 units
  int *part_count;      // [num_seqs * gx * num_kv_heads] pieces finished per item
  int32_t *ws_err;      // the workspace's error word
  // the step's cache write folded into the launch (pa_mixed_attention_append,
  // 16-bit caches, chunk mode): the new K/V rows of the chunks, row
  // query_start_loc[s] + i for query i of sequence s, as [rows][kv heads][D]
  // (box {64, 1, 16}: 16 consecutive tokens of one kv head).  Keys at or past
  // a chunk's first position come from these rows, not from the caches, and
  // every tile writes its own queries' rows into the caches (k_write,
  // v_write).  Each chunk starts at a block boundary (checked).
  CUtensorMap knmap;
  CUtensorMap vnmap;
  int new_rows;         // 1: the above applies
  int64_t new_row_count;  // rows of k_new / v_new (of the prefill part)
  const uint8_t *k_new;
  const uint8_t *v_new;
  uint8_t *k_write;
  uint8_t *v_write;
};

// One call of prefill_tile: the item (sequence s, key split, kv head,
// query tile) and the part of its KV iterations that this call covers.  A
// piece of an item cut between the CTAs of a balanced launch also carries
// where the item's other pieces are.
struct Seg {
  int s, split, kvh, qtile, gx;
  int it_lo, it_hi;       // KV iterations [it_lo, it_hi) of the item; it_hi < 0: all
  int piece;              // 1: the item is cut between CTAs c_lo .. c_hi
  int slot;               // this piece's slot
  int item;               // the item's piece counter
  int c_lo, c_hi, me, G;  // CTAs holding the pieces; this CTA; CTAs sharing the work
  int item_start;         // the item's first unit
  int U;                  // units of the launch (below 2^31)
};

// CTA c of G takes units [c U / G, (c + 1) U / G); cta_of(u) is the CTA
// holding unit u, and a piece's slot is 0 for the CTA's first item (the item
// began at or before the CTA's first unit) and 1 for its last.
__device__ __forceinline__ int sk_first_unit(int c, int U, int G) {
  return static_cast<int>(static_cast<long long>(c) * U / G);
}
__device__ __forceinline__ int sk_cta_of(int u, int U, int G) {
  return static_cast<int>((static_cast<long long>(u + 1) * G - 1) / U);
}
__device__ __forceinline__ int sk_slot(int c, int item_start, int U, int G) {
  return c * 2 + (item_start <= sk_first_unit(c, U, G) ? 0 : 1);
}

// The queries and keys of one item.  False if it has no query (or a
// checked length was bad: its rows are then left unwritten); a checked
// length out of range is reported if report is set.
struct ItemRange {
  int qs, q_len, L, qt0, nq, p_lo, p_hi, base_pos, kv_end, kv_lo, j0, n_tiles;
};
__device__ __forceinline__ bool item_range(const Args &a, int s, int split, int qtile, int gx, bool report,
                                           ItemRange &r) {
  r.qs = __ldg(a.query_start_loc + s);
  r.q_len = __ldg(a.query_start_loc + s + 1) - r.qs;
  r.L = __ldg(a.context_lens + s);
  if (a.checked) {
    // lengths within the table's capacity; a chunk no longer than its context
    // nor than the launch's query tiles; rows start at a row >= 0
    int32_t *e1 = report ? a.err : nullptr, *e2 = report ? a.ws_err : nullptr;
    r.L = checked_len(r.L, a.max_blocks_per_seq * 16, e1, e2);
    r.q_len = checked_len(r.q_len, a.prefix_mode ? gx * a.qt : min(r.L, gx * a.qt), e1, e2);
    if (r.qs < 0) {
      if (report && threadIdx.x == 0) report_error(a.err, a.ws_err, kErrBadIndex);
      return false;
    }
  }
  r.qt0 = qtile * a.qt;
  if (r.qt0 >= r.q_len) return false;
  r.nq = min(a.qt, r.q_len - r.qt0);
  // prefix mode: the split covers prefix keys [p_lo, p_hi), and every query
  // comes after them all; otherwise query i sits at L - q_len + i
  r.p_lo = a.prefix_mode ? min(r.L, split * a.split_len) : 0;
  r.p_hi = a.prefix_mode ? min(r.L, r.p_lo + a.split_len) : 0;
  r.base_pos = a.prefix_mode ? r.p_hi - 1 : r.L - r.q_len + r.qt0;  // position of query qt0
  r.kv_end = a.prefix_mode ? r.p_hi : r.base_pos + r.nq;            // keys [kv_lo, kv_end) are needed
  // local attention: the earliest query sees keys from kv_lo on (the first
  // key never decreases with the position)
  r.kv_lo = a.prefix_mode ? r.p_lo : local_first_key(r.base_pos, a.window, a.chunk);
  r.j0 = r.kv_lo / KT;
  r.n_tiles = (r.kv_end + KT - 1) / KT;
  return true;
}

// KV iterations of pair p's items (chunk mode), 0 if it has no query
__device__ __forceinline__ int pair_iters(const Args &a, int p) {
  ItemRange r;
  if (!item_range(a, p / a.gx, 0, a.gx - 1 - p % a.gx, a.gx, false, r)) return 0;
  return max(0, r.n_tiles - r.j0);
}

// Optional timeline counters (compiled only with -DPA_PREFILL_TRACE), per
// CTA slot (blockIdx linearised, first 4096): softmax warp 0 lane 0 cycles
// [0] waiting for S, [1] loading S, masking and max, [2] rescaling O, [3]
// exp2 and P stores, [4] fence and arrive, [7] total; MMA thread cycles [8]
// waiting for V, [9] waiting for K, [10] waiting for P, [11] total;
// producer [12] waiting for free slots, [13] total; [14] KV tiles.
// Optional event timeline of CTA (0, 0, 0) (compiled only with
// -DPA_PREFILL_TIMELINE): clock64 per KV tile j of [0] P_A seen by the MMA
// thread, [1] PV_A + QK_A issued, [2] P_B seen, [3] PV_B + QK_B issued,
// [4] S_A seen by softmax A, [5] P_A arrived, [6] S_B seen, [7] P_B arrived,
// [8 + w] softmax warp w arrived, [16] V of the next tile seen by the MMA
// thread, [17] V landed as seen by converter thread 0, [18] V converted
// (fp16 P), [19] start of the MMA thread's V wait,
// softmax A: [20] after the fence, [21] first scores loaded, [22] chunks
// done, [23] stores done.
#ifdef PA_PREFILL_TIMELINE
static __device__ long long g_pf_tl[24][64];
#define PF_TL(i, j) \
  if (blockIdx.x == 0 && blockIdx.y == 0 && blockIdx.z == 0 && (j) < 64) g_pf_tl[i][j] = clock64()
#else
#define PF_TL(i, j)
#endif
#ifdef PA_PREFILL_TRACE
static __device__ unsigned long long g_pf_trace[4096][16];
#define PF_TRACE(...) __VA_ARGS__
#else
#define PF_TRACE(...)
#endif

// How O += P V runs (see the file comment):
//   kPvPair  P as a hi + lo pair of the cache's 16-bit type, V as cached
//   kPvF16   P as one fp16 value, V in fp16 (a bf16 V tile is converted in
//            shared memory by warps 2-3)
constexpr int kPvPair = 0;
constexpr int kPvF16 = 1;

template <int D, int KVT, int PVM>
struct Cfg {
  static constexpr bool P16 = PVM == kPvF16;           // single fp16 P
  static constexpr bool CONVERT = P16 && KVT == kKvBf16;  // V tiles converted bf16 -> fp16
  // 8-bit caches (E4M3, E5M2): K and V tiles land as bytes in the second
  // half of their slot and are widened in place to fp16 (exact); Q is staged
  // in fp16, so both products take fp16 operands
  static constexpr bool KV8 = !kv16(KVT);
  static constexpr bool F16OPS = KVT == kKvF16 || KV8;  // QK in fp16
  static_assert(!KV8 || (P16 && D == 128), "8-bit caches: fp16 P, head_dim 128");
  static constexpr int HALVES = D / 64;          // 128-byte column halves of a row
  static constexpr int QHALF = MT * 128;         // bytes of one half of one Q tile
  static constexpr int QB = HALVES * QHALF;      // one Q tile
  static constexpr int KVHALF = KT * 128;        // bytes of one half of a K or V tile
  static constexpr int KVB = HALVES * KVHALF;
  static constexpr int OFF_Q = 0;                  // [NQT]
  static constexpr int OFF_K = OFF_Q + NQT * QB;   // [NSK]
  static constexpr int OFF_V = OFF_K + NSK * KVB;  // [NSV]
  static constexpr int OFF_BAR = OFF_V + NSV * KVB;
  static constexpr int OFF_X = OFF_BAR + 256;          // softmax exchange: [2][MT] fp32
  static constexpr int OFF_M = OFF_X + 2 * MT * 4;     // balanced launch: merges this CTA owes (128 B)
  static constexpr int SMEM = OFF_M + 128 + 1024;      // + 1024-B alignment slack
  // at least half an SM's shared memory, so that two CTAs (each holding
  // all 512 TMEM columns) never share an SM
  static constexpr int SMEM_LAUNCH = SMEM > 120 * 1024 ? SMEM : 120 * 1024;
  static_assert(SMEM <= 232448, "shared memory of one CTA");
  // TMEM columns: S_t of each Q tile (KT each; P_t hi | lo written over it),
  // then O_t (D each)
  static constexpr uint32_t O_COL = NQT * KT;
  static constexpr uint32_t TMEM_COLS = 512;
  static_assert(NQT * (KT + D) <= TMEM_COLS, "TMEM columns");
  static constexpr uint32_t IDESC_QK = umma_idesc_bf16(MT, KT, false, false, F16OPS);
  static constexpr uint32_t IDESC_PV = umma_idesc_bf16(MT, D, false, true, P16 || KVT == kKvF16);
  // bytes landed per 16-token block of K (or of V), all halves
  static constexpr uint32_t BLOCK_BYTES = KV8 ? 16u * D : HALVES * 16u * 128u;
};

// barriers: K_FULL[NSK], K_EMPTY[NSK], V_FULL[NSV], V_EMPTY[NSV],
// S_FULL[tile], P_FULL[tile], V_READY[NSV] (fp16 P: the V tile is in fp16,
// rows outside the needed keys zeroed), K_READY[NSK] (8-bit caches: the K
// tile widened to fp16), Q_FULL (the Q tiles that come by TMA), Q_EMPTY
enum Bar {
  K_FULL = 0,
  K_EMPTY = K_FULL + NSK,
  V_FULL = K_EMPTY + NSK,
  V_EMPTY = V_FULL + NSV,
  S_FULL = V_EMPTY + NSV,
  P_FULL = S_FULL + NQT,
  V_READY = P_FULL + NQT,
  K_READY = V_READY + NSV,  // 8-bit caches: the K tile widened to fp16
  Q_FULL = K_READY + NSK,   // the Q tiles copied by TMA have landed
  Q_EMPTY = Q_FULL + 1,     // balanced launch: a segment's last QKs completed (Q may be replaced)
  NBAR = Q_EMPTY + 1
};
static_assert(NBAR * 8 + 24 <= 256, "barriers, TMEM slot and flags fit their 256 bytes");

// Shared memory of a CTA: the tile's operands at 1024-byte alignment, then
// its barriers, the TMEM slot and three flags (see Cfg::OFF_BAR).
__device__ __forceinline__ uint8_t *align1024(uint8_t *p) {
  return reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(p) + 1023) & ~uintptr_t(1023));
}

// One prefill tile: the item of sg (its KV iterations [it_lo, it_hi)).  Run
// by all NTHREADS threads of a CTA with tensor memory already allocated
// (tmem: all TMEM_COLS columns); every thread takes the same early returns.
// On return every copy and product of the tile has completed, so that its
// barriers can be set up again for the next tile.  NR: compiled with the
// fused cache write of a step (Args::new_rows), which only the single-launch
// step uses; the other kernels are built without it.
template <int D, int KVT, int PVM, bool NR = false>
__device__ void prefill_tile(const Args &a, uint8_t *smem, uint32_t tmem, const Seg &sg) {
  using C = Cfg<D, KVT, PVM>;
  uint64_t *bar = reinterpret_cast<uint64_t *>(smem + C::OFF_BAR);
  uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(bar + NBAR);
  int *s_abort = reinterpret_cast<int *>(tmem_slot + 1);
  int *s_last_k = s_abort + 1;  // last KV tile whose K copies the producer issued
  int *s_last_v = s_abort + 2;  // ... and whose V copies

  const int split = sg.split;
  const int s = sg.s;
  const int kvh = sg.kvh;
  // where the first key is 0 (chunk mode, no local attention, the item's
  // first tile), the producer loads the first tile's block ids at once,
  // beside the lengths instead of after them
  const bool spec_ok = !a.prefix_mode && a.window == 0 && a.chunk == 0 && sg.it_lo == 0;
  int spec = 0;
  {
    constexpr int BOXES = C::KV8 ? 1 : C::HALVES;
    const int l = threadIdx.x & 31, b = l / BOXES;
    if (spec_ok && (threadIdx.x >> 5) == kProducerWarp && l < BPT * BOXES && b < a.max_blocks_per_seq)
      spec = __ldg(a.block_tables + static_cast<int64_t>(s) * a.max_blocks_per_seq + b);
  }
  ItemRange ir;
  if (!item_range(a, s, split, sg.qtile, sg.gx, true, ir)) return;
  const int qs = ir.qs;
  const int qt0 = ir.qt0;
  const int nq = ir.nq;
  const int p_lo = ir.p_lo;
  const int p_hi = ir.p_hi;
  const int base_pos = ir.base_pos;
  const int kv_end = ir.kv_end;
  // the chunk's new rows are read from the step's new K/V (a fused cache
  // write).  chunk0 is the position of the chunk's first query (base_pos is
  // that of this tile's first query, qt0 queries later); it must start a
  // block, or the block it falls in would hold new rows not yet in the cache
  const bool new_src = NR && !C::KV8 && a.new_rows && !a.prefix_mode;
  const int chunk0 = base_pos - qt0;
  if (new_src && (chunk0 & 15) != 0 && threadIdx.x == 0) report_error(a.err, a.ws_err, kErrBadIndex);
  if (a.prefix_mode && p_hi <= p_lo) {
    // no key in this split (an empty or short shared prefix): out = 0,
    // lse = -inf, before any barrier or tensor memory is set up
    for (int i = threadIdx.x; i < nq * a.g; i += NTHREADS) {
      const int64_t row =
          (static_cast<int64_t>(qs + qt0 + i / a.g) * a.num_q_heads + kvh * a.g + i % a.g) * a.out_slots + split;
      for (int d = 0; d < D; d += 4) *reinterpret_cast<float4 *>(a.out + row * D + d) = make_float4(0.f, 0.f, 0.f, 0.f);
      if (a.lse) a.lse[row] = -INFINITY;
    }
    return;
  }
  // KV tiles j0 .. j0 + n_iter - 1 are walked (the item's iterations
  // [it_lo, it_hi)); the rings and barriers count iterations jj = j - j0
  const int kv_lo = ir.kv_lo;
  const int it_hi = sg.it_hi < 0 ? ir.n_tiles - ir.j0 : sg.it_hi;
  const int j0 = ir.j0 + sg.it_lo;
  const int n_iter = it_hi - sg.it_lo;
  const int tid = threadIdx.x;
  const int warp = tid >> 5;
  const int lane = tid & 31;
  const int g = a.g;
  const int rows_used = a.qt * g;

  if (tid == 0) {
    for (int i = 0; i < NSK; ++i) {
      mbar_init(&bar[K_FULL + i], 1);
      mbar_init(&bar[K_EMPTY + i], 1);
    }
    for (int i = 0; i < NSV; ++i) {
      mbar_init(&bar[V_FULL + i], 1);
      mbar_init(&bar[V_EMPTY + i], 1);
    }
    for (int t = 0; t < NQT; ++t) {
      mbar_init(&bar[S_FULL + t], 1);
      mbar_init(&bar[P_FULL + t], 8);
    }
    for (int i = 0; i < NSV; ++i) mbar_init(&bar[V_READY + i], 2);
    for (int i = 0; i < NSK; ++i) mbar_init(&bar[K_READY + i], 2);
    mbar_init(&bar[Q_FULL], 1);
    *s_abort = 0;
    *s_last_k = -1;
    *s_last_v = -1;
    fence_mbar_init();
  }

  // ---- Q tiles: row R = query * g + head (tile R / 128, lane R % 128),
  // [tile][half][row][128 B], 128-B swizzle.  A tile whose 128 / g queries
  // all belong to the chunk comes by TMA (16-bit caches, g dividing 128):
  // the box's rows are its queries times the g heads of the kv head, in
  // the order of R.  The producer issues those copies at once and goes on
  // to the K/V copies; the MMA thread waits for them (Q_FULL).  Every other
  // tile is staged by the threads (rows past the chunk zeroed).  With an
  // 8-bit cache the bf16 queries are staged as fp16 (round to nearest; a
  // finite |q| >= 2^16 does not fit and is reported).
  uint32_t qtma_tiles = 0;
  if (!C::KV8 && a.qtma) {
#pragma unroll
    for (int t = 0; t < NQT; ++t)
      if ((t + 1) * (MT / g) <= nq) qtma_tiles |= 1u << t;
  }
  const int32_t *table = a.block_tables + static_cast<int64_t>(s) * a.max_blocks_per_seq;
  // producer: lane -> (block of the tile, half); the same lanes copy K and
  // V.  An 8-bit block is one box of 16 rows of D bytes, landing in the
  // second half of the slot (widened in place by warps 2-3)
  constexpr int BOXES = C::KV8 ? 1 : C::HALVES;
  const int bi = lane / BOXES;
  const int hh = lane % BOXES;
  const bool issuer = lane < BPT * BOXES;
  auto block_id = [&](int lb) {
    const int v = __ldg(table + lb);
    return a.checked ? checked_block(v, a.num_blocks, a.err, a.ws_err) : v;
  };
  int phys_next = 0;
  if (qtma_tiles != 0) __syncthreads();  // the barriers are set up
  if (warp == kProducerWarp) {
    // the first KV tile's block ids load while Q is set up
    if (issuer && (j0 * BPT + bi) * 16 < kv_end)
      phys_next = spec_ok ? (a.checked ? checked_block(spec, a.num_blocks, a.err, a.ws_err) : spec)
                          : block_id(j0 * BPT + bi);
    if (qtma_tiles != 0 && lane == 0 && !a.stall) {
      const uint64_t pol = l2_evict_first_policy();
      mbar_arrive_expect_tx(&bar[Q_FULL], __popc(qtma_tiles) * C::QB);
#pragma unroll
      for (int t = 0; t < NQT; ++t)
        if (qtma_tiles >> t & 1)
#pragma unroll
          for (int q2 = 0; q2 < C::HALVES; ++q2)
            tma_load_3d(smem + C::OFF_Q + t * C::QB + q2 * C::QHALF, &a.qmap, q2 * 64, kvh * g,
                        qs + qt0 + t * (MT / g), &bar[Q_FULL], pol);
    }
  }
  if (qtma_tiles != (1u << NQT) - 1) {
    constexpr int CHUNKS = D / 8;  // 16-byte chunks per row
    float qmax = 0.f;
    for (int i = tid; i < MROWS * CHUNKS; i += NTHREADS) {
      const int R = i / CHUNKS;
      if (qtma_tiles >> (R / MT) & 1) continue;
      const int ch = i - R * CHUNKS;
      const int qi = R / g;
      const bool ok = R < rows_used && qi < nq;
      const uint16_t *src = a.q;
      if (ok) src = a.q + (static_cast<int64_t>(qs + qt0 + qi) * a.num_q_heads + kvh * g + (R - qi * g)) * D + ch * 8;
      const int r = R & (MT - 1);
      uint8_t *dst = smem + C::OFF_Q + (R / MT) * C::QB + (ch >> 3) * C::QHALF + r * 128 + (((ch & 7) ^ (r & 7)) << 4);
      if constexpr (C::KV8) {
        uint4 y = make_uint4(0, 0, 0, 0);
        if (ok) {
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
        cp_async16(dst, src, ok);
      }
    }
    if (C::KV8 && qmax >= 65536.f && qmax <= FLT_MAX) report_error(a.err, a.ws_err, kErrFp16Range);
    cp_async_commit();
    cp_async_wait<0>();
    fence_proxy_async_smem();
  }
  tc_fence_before_sync();
  __syncthreads();
  tc_fence_after_sync();
  const uint32_t sbase = smem_u32(smem);

  if (warp == kProducerWarp) {
    // ------------------------------------------------------ TMA producer
    const uint64_t pol = l2_evict_first_policy();
    PF_TRACE(const long long tp0 = clock64(); long long tp_wait = 0;)
    bool ok = true;
    // test hook: issue nothing and signal nothing, so the other warps' waits
    // run out with nothing in flight
    for (int jj = 0; jj < (a.stall ? 0 : n_iter) && ok; ++jj) {
      const int j = j0 + jj;
      const int phys = phys_next;
      const int key0 = j * KT;
      const int lb = (j + 1) * BPT + bi;  // prefetch the next tile's block id
      phys_next = (issuer && lb * 16 < kv_end) ? block_id(lb) : 0;
      const int nblk = min(BPT, (kv_end - key0 + 15) / 16);
      // blocks of the first tile entirely before the item's first key are
      // not read (under local attention their pages may be gone); a piece
      // that starts later has none
      const int bskip = jj == 0 ? max(0, (kv_lo >> 4) - j * BPT) : 0;
      const int row = (phys * a.num_kv_heads + kvh) * 16;
      // K of tile j (its slot frees once the QKs of tile j - NSK completed),
      // then V of tile j (once the PVs of tile j - NSV completed)
#pragma unroll 1
      for (int part = 0; part < 2; ++part) {
        const int st = part ? jj % NSV : jj % NSK;
        const uint32_t ph = part ? (jj / NSV) & 1 : (jj / NSK) & 1;
        const int full = (part ? V_FULL : K_FULL) + st;
        PF_TRACE(const long long tw = clock64();)
        if (!mbar_wait(&bar[(part ? V_EMPTY : K_EMPTY) + st], ph ^ 1, a.wait_ns)) {
          ok = false;
          break;
        }
        PF_TRACE(tp_wait += clock64() - tw;)
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
          const int lpos0 = key0 + bi * 16;  // the block's first position
          if (NR && !C::KV8 && new_src && lpos0 >= chunk0)
            // a block of the chunk's own new tokens (query lpos0 - chunk0
            // onwards): from the step's new rows
            tma_load_3d(dst, part ? &a.vnmap : &a.knmap, hh * 64, kvh, qs + (lpos0 - chunk0), &bar[full], pol);
          else
            tma_load_2d(dst, part ? &a.vmap : &a.kmap, hh * 64, row, &bar[full], pol);
        }
        if (lane == 0) *(part ? s_last_v : s_last_k) = jj;
      }
    }
    if (!ok && lane == 0) *s_abort = 1;
    PF_TRACE(const int slot = (blockIdx.z * gridDim.y + blockIdx.y) * gridDim.x + blockIdx.x;
             if (lane == 0 && slot < 4096) { g_pf_trace[slot][12] = tp_wait; g_pf_trace[slot][13] = clock64() - tp0; g_pf_trace[slot][14] = n_iter; })
  } else if (warp == kMmaWarp) {
    // --------------------------------------------------------- MMA issuer
    if (lane == 0) {
      bool ok = true;
      auto qk = [&](int t, int jj) {  // S_t = Q_t K^T of iteration jj
        const uint32_t qbase = sbase + C::OFF_Q + t * C::QB;
        const uint32_t kbase = sbase + C::OFF_K + (jj % NSK) * C::KVB;
#pragma unroll
        for (int kk = 0; kk < D / 16; ++kk) {
          const uint64_t ad = umma_desc_sw128(qbase + (kk >> 2) * C::QHALF + (kk & 3) * 32, 16, 1024);
          const uint64_t bd = umma_desc_sw128(kbase + (kk >> 2) * C::KVHALF + (kk & 3) * 32, 16, 1024);
          umma_bf16_ss(tmem + t * KT, ad, bd, C::IDESC_QK, kk > 0 ? 1u : 0u);
        }
      };
      auto pv = [&](int t, int jj) {  // O_t += P_t V of iteration jj, P_t from TMEM
        const uint32_t vbase = sbase + C::OFF_V + (jj % NSV) * C::KVB;
        constexpr int NPART = C::P16 ? 1 : 2;  // fp16 P, or the hi and lo halves of a pair
#pragma unroll
        for (int part = 0; part < NPART; ++part) {
#pragma unroll
          for (int kk = 0; kk < KT / 16; ++kk) {
            // keys 16 kk .. 16 kk + 15: chunk kk / 2 (P, or hi at +0 and lo at +16)
            const uint64_t bd = umma_desc_sw128(vbase + kk * 2048, C::KVHALF, 1024);
            umma_bf16_ts(tmem + C::O_COL + t * D, tmem + t * KT + (kk >> 1) * 32 + part * 16 + (kk & 1) * 8, bd,
                         C::IDESC_PV, (jj > 0 || part > 0 || kk > 0) ? 1u : 0u);
          }
        }
      };
      PF_TRACE(const long long tm0 = clock64(); long long tm_v = 0, tm_k = 0, tm_p = 0; long long tw;)
      // Issue order per KV tile j: PV_A(j), QK_A(j+1), S_A commit, K_EMPTY(j)
      // commit, PV_B(j), V_EMPTY(j) commit, wait for V(j+1), QK_B(j+1), S_B
      // commit.  The tensor pipe queues only a few instructions, so buffer
      // releases and the V wait sit between MMAs (while the pipe has work)
      // and the thread goes straight from the last MMA of a KV tile to the
      // wait for the next tile's P_A.
      // V is ready for the MMAs once it landed (pair mode) or once warps 2-3
      // converted it (fp16 P)
      constexpr int VB = C::P16 ? V_READY : V_FULL;
      constexpr int KB = C::KV8 ? K_READY : K_FULL;  // 8-bit: once widened to fp16
      // the first QKs need Q and K only; V of the first tile (and its
      // conversion) is waited for behind them
      if ((qtma_tiles != 0 && !mbar_wait(&bar[Q_FULL], 0, a.wait_ns)) || !mbar_wait(&bar[KB], 0, a.wait_ns))
        ok = false;
      if (ok) {
        tc_fence_after_sync();
        for (int t = 0; t < NQT; ++t) {
          qk(t, 0);
          umma_commit(&bar[S_FULL + t]);
        }
        if (!mbar_wait(&bar[VB], 0, a.wait_ns)) ok = false;
      }
      for (int jj = 0; jj < n_iter && ok; ++jj) {
        const bool next = jj + 1 < n_iter;
        for (int t = 0; t < NQT; ++t) {
          if (!mbar_wait_hint(&bar[P_FULL + t], jj & 1, a.wait_ns)) {
            ok = false;
            break;
          }
          PF_TL(t * 2, jj);
          tc_fence_after_sync();
          pv(t, jj);
          if (t == NQT - 1) {
            umma_commit(&bar[V_EMPTY + jj % NSV]);  // both tiles are done with V of iteration jj
            PF_TL(19, jj);
            if (next && !mbar_wait(&bar[VB + (jj + 1) % NSV], ((jj + 1) / NSV) & 1, a.wait_ns)) {
              ok = false;
              break;
            }
            PF_TL(16, jj);
          }
          if (next) {
            if (t == 0) {
              if (!mbar_wait(&bar[KB + (jj + 1) % NSK], ((jj + 1) / NSK) & 1, a.wait_ns)) {
                ok = false;
                break;
              }
            }
            tc_fence_after_sync();
            qk(t, jj + 1);
          }
          // S_t of the next KV tile is ready and PV_t(jj) has completed
          // (after the last tile: O_t is final)
          umma_commit(&bar[S_FULL + t]);
          if (t == 0) umma_commit(&bar[K_EMPTY + jj % NSK]);  // both tiles are done with K of iteration jj
          PF_TL(t * 2 + 1, jj);
        }
      }
      if (!ok) *s_abort = 1;
      PF_TRACE(const int slot = (blockIdx.z * gridDim.y + blockIdx.y) * gridDim.x + blockIdx.x;
               if (slot < 4096) { g_pf_trace[slot][8] = tm_v; g_pf_trace[slot][9] = tm_k; g_pf_trace[slot][10] = tm_p; g_pf_trace[slot][11] = clock64() - tm0; })
    }
    __syncwarp();
  } else if (C::P16 && warp >= kConvWarp0 && warp < kConvWarp0 + 2) {
    // --------------------------------- K / V tile preparation (fp16 P)
    // Each landed V tile: rows outside the needed keys [kv_lo, kv_end)
    // zeroed (stale or poisoned data; 0 * NaN would not vanish in the PV),
    // and for a bf16 cache every element converted to fp16 in place (round
    // to nearest; exact for |v| in [2^-14, 2^16), within 2^-25 below).  A
    // finite |v| >= 2^16 does not fit fp16: it is reported
    // (PA_DEVERR_FP16_RANGE) and its products are wrong.  With an 8-bit
    // cache the K tile is widened to fp16 as well (exact).  The MMA issuer
    // waits for V_READY (and K_READY).
    const int ct = tid - kConvWarp0 * 32;
    bool ok = true;
    float vmax = 0.f;
    constexpr int UNITS = C::KVB / 16;   // 16-byte units of a V tile
    constexpr int UROW = KT * 8;         // units of one 128-byte column half
    // 8-bit caches: widen the tile of a slot in place.  The bytes landed in
    // the slot's second half as rows of 128 bytes (16-byte chunk c of row r
    // at (c ^ (r & 7)) * 16, the TMA's 128-byte swizzle); the fp16 tile
    // takes the whole slot as [half][row][128 B], same swizzle.  Dims 0-63
    // (chunks 0-3) go to the first half, which the bytes do not occupy;
    // dims 64-127 are read first, then (after a barrier of the two
    // converter warps) written over them.  Rows outside [r_lo, r_hi) become
    // zero where zero_rows is set (V: 0 * NaN would not vanish).
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
        const int k0 = 2 * c4, k1 = 2 * c4 + 1;  // output chunks of 8 fp16
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
    for (int jj = 0; jj < n_iter; ++jj) {
      const int key0 = (j0 + jj) * KT;
      const int r_lo = max(kv_lo - key0, 0);
      const int r_hi = min(kv_end - key0, KT);
      if constexpr (C::KV8) {
        // K of this tile first (the MMAs need it before V); both warps agree
        // to go on, so their barrier in widen8 stays matched
        const int stk = jj % NSK;
        if (!named_bar_and(2, 64, mbar_wait(&bar[K_FULL + stk], (jj / NSK) & 1, a.wait_ns))) {
          ok = false;
          break;
        }
        widen8(smem + C::OFF_K + stk * C::KVB, r_lo, r_hi, false);
        fence_proxy_async_smem();
        __syncwarp();
        if (lane == 0) mbar_arrive(&bar[K_READY + stk]);
      }
      const int st = jj % NSV;
      if (!named_bar_and(2, 64, mbar_wait(&bar[V_FULL + st], (jj / NSV) & 1, a.wait_ns))) {
        ok = false;
        break;
      }
      if (ct == 0) PF_TL(17, jj);
      uint4 *vt = reinterpret_cast<uint4 *>(smem + C::OFF_V + st * C::KVB);
      if constexpr (C::KV8) {
        widen8(smem + C::OFF_V + st * C::KVB, r_lo, r_hi, true);
      } else if constexpr (C::CONVERT) {
        // eight 16-byte units per step, all loads issued before any
        // conversion so that their latencies overlap
        constexpr int ILP = 8;
        static_assert(UNITS % (64 * ILP) == 0, "whole steps");
#pragma unroll 1
        for (int u0 = ct; u0 < UNITS; u0 += 64 * ILP) {
          uint4 x[ILP];
#pragma unroll
          for (int k = 0; k < ILP; ++k) x[k] = vt[u0 + 64 * k];
#pragma unroll
          for (int k = 0; k < ILP; ++k) {
            const int row = ((u0 + 64 * k) % UROW) >> 3;  // [half][row][128 B]
            const uint32_t w[4] = {x[k].x, x[k].y, x[k].z, x[k].w};
            uint32_t y[4];
            float um = 0.f;
#pragma unroll
            for (int e = 0; e < 4; ++e) {
              const float f0 = bf16lo(w[e]), f1 = bf16hi(w[e]);
              um = fmaxf(um, fmaxf(fabsf(f0), fabsf(f1)));
              y[e] = pack_f16x2(f0, f1);
            }
            // rows outside the needed keys hold anything: zeroed, not checked
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
      if (ct == 0) PF_TL(18, jj);
    }
    // finite values beyond fp16's range (NaN is skipped by fmaxf; an
    // infinity propagates as it does in exact arithmetic)
    if (C::CONVERT && vmax >= 65536.f && vmax <= FLT_MAX) report_error(a.err, a.ws_err, kErrFp16Range);
    if (!ok && lane == 0) *s_abort = 1;
  } else if (warp >= kSoftmaxWarp0) {
    // ------------------------------------- softmax, two threads per row
    // Warps 4-7 take keys 0-63 and warps 8-11 keys 64-127 of every KV tile,
    // for Q tile A and then for Q tile B (the order the MMAs produce them),
    // so two softmax warps per SM sub-partition share each tile.  A thread
    // holds row r = 32 (warp % 4) + lane (its TMEM lane) and its half h of
    // the keys.  The two threads of a row exchange their maxima through
    // shared memory, so the tile's row maximum is known before any P is
    // written: a rise of the running maximum rescales O (each thread its
    // half of the columns) and never P.  Only partner warps w and w + 4 (the
    // same rows) exchange anything, so each pair has its own named barrier
    // (3 + w % 4, 64 threads) and never waits for the other pairs.
    const int h = (warp - kSoftmaxWarp0) >> 2;  // half of the keys
    const int r = ((warp & 3) << 5) | lane;     // row of a Q tile = TMEM lane
    const uint32_t trow = tmem + (static_cast<uint32_t>((warp & 3) * 32) << 16);
    float *xch = reinterpret_cast<float *>(smem + C::OFF_X);  // [2][MT] maxima / sums of the halves
    const int pair_bar = 3 + (warp & 3);  // named barrier of this partner pair (64 threads)
    // score scale and output scale of this kv head (its own k / v scale
    // where an 8-bit cache has per-head scales)
    const float qscale = a.k_scales ? a.qscale0 * __ldg(a.k_scales + kvh) : a.qscale;
    const float vscale = a.v_scales ? __ldg(a.v_scales + kvh) : a.vscale;
    float m_ref[NQT], l[NQT];
    int pos[NQT], first[NQT];
#pragma unroll
    for (int t = 0; t < NQT; ++t) {
      const int R = t * MT + r;
      const int qi = R / g;
      const bool rv = R < rows_used && qi < nq;
      pos[t] = rv ? (a.prefix_mode ? base_pos : base_pos + qi) : -1;  // keys <= pos are visible
      first[t] = a.prefix_mode ? kv_lo : local_first_key(pos[t], a.window, a.chunk);  // ... and keys >= first
      m_ref[t] = -INFINITY;
      l[t] = 0.f;
    }
    if constexpr (NR && !C::KV8) {
      if (new_src) {
        // the fused cache write: this tile's queries' new K and V rows (of
        // its kv head) into the caches, before the first scores arrive.  In
        // this launch nothing reads those cache rows: every tile takes the
        // chunk's keys from the new rows.  Four tasks per query (K or V, half
        // a row each), 16-byte vectors.
        constexpr int NV = D / 16;  // vectors per half row
        const int st0 = tid - kSoftmaxWarp0 * 32;
        for (int task = st0; task < nq * 4; task += 256) {
          const int qi = task >> 2, isv = (task >> 1) & 1, half = task & 1;
          const int pos = base_pos + qi;  // query qt0 + qi of the chunk
          int phys = __ldg(table + (pos >> 4));
          if ((a.checked && (phys < 0 || phys >= a.num_blocks)) || qs + qt0 + qi >= a.new_row_count) {
            // nothing written outside the cache, nothing read past the new rows
            report_error(a.err, a.ws_err, kErrBadIndex);
            continue;
          }
          const uint4 *src = reinterpret_cast<const uint4 *>(
                                 (isv ? a.v_new : a.k_new) +
                                 (static_cast<int64_t>(qs + qt0 + qi) * a.num_kv_heads + kvh) * (D * 2)) +
                             half * NV;
          uint4 *dst = reinterpret_cast<uint4 *>(
                           (isv ? a.v_write : a.k_write) +
                           ((static_cast<int64_t>(phys) * a.num_kv_heads + kvh) * 16 + (pos & 15)) * (D * 2)) +
                       half * NV;
          uint4 v[NV];
#pragma unroll
          for (int i = 0; i < NV; ++i) v[i] = __ldg(src + i);
#pragma unroll
          for (int i = 0; i < NV; ++i) dst[i] = v[i];
        }
      }
    }
    bool ok = true;
    PF_TRACE(const long long ts0 = clock64(); long long tq[7] = {0, 0, 0, 0, 0, 0, 0}; long long tc, tk;)
    for (int jj = 0; jj < n_iter && ok; ++jj) {
      const int j = j0 + jj;
      const int key0 = j * KT;
#pragma unroll
      for (int t = 0; t < NQT; ++t) {
        PF_TRACE(tc = clock64();)
        bool got = mbar_wait_hint(&bar[S_FULL + t], jj & 1, a.wait_ns);
        PF_TRACE(tq[0] += clock64() - tc; tc = clock64();)
        if (r == 0 && h == 0) PF_TL(4 + t * 2, jj);
        tc_fence_after_sync();
        const uint32_t s_col = t * KT;
        const uint32_t o_col = C::O_COL + t * D;
        if (!C::P16 && t == 0 && h == 0 && jj == n_iter - 1 && kv_end - key0 < KT && got) {
          // pair mode: V rows past the last needed key are zeroed (stale or
          // poisoned data), after this tile's V copies landed; tile 0's PV
          // of this KV tile is issued before tile 1's
          got = mbar_wait(&bar[V_FULL + jj % NSV], (jj / NSV) & 1, a.wait_ns);
          const int kval = kv_end - key0;
          for (int i = r; got && i < (KT - kval) * C::HALVES * 8; i += MT) {
            const int row = kval + i / (C::HALVES * 8);
            const int rem = i % (C::HALVES * 8);
            *reinterpret_cast<uint4 *>(smem + C::OFF_V + (jj % NSV) * C::KVB + (rem >> 3) * C::KVHALF + row * 128 +
                                       (rem & 7) * 16) = make_uint4(0, 0, 0, 0);
          }
          fence_proxy_async_smem();
        }
        // both warps of the pair go on, or both stop (a bounded wait ran
        // out): the pair's named barriers below stay matched.  This barrier also tells a
        // thread that its partner has read the previous exchange.
        if (!named_bar_and(pair_bar, 64, got)) {
          ok = false;
          break;
        }
        // this half's 64 scores: TMEM chunks 2h and 2h + 1 (32 keys each)
        uint32_t sc[2][32];
        tmem_ld32_async(trow + s_col + (2 * h) * 32, sc[0]);
        tmem_ld32_async(trow + s_col + (2 * h + 1) * 32, sc[1]);
        tmem_wait_ld(sc[0]);
        tmem_wait_ld(sc[1]);
        PF_TRACE(tq[1] += clock64() - tc; tc = clock64();)
        const int kh = key0 + h * 64;  // first key of this half
        float mx = -INFINITY;
#pragma unroll
        for (int c = 0; c < 2; ++c) {
          const int kc = kh + c * 32;
          if (!(kc + 31 <= pos[t] && kc >= first[t])) {
#pragma unroll
            for (int i = 0; i < 32; ++i)
              if (kc + i > pos[t] || kc + i < first[t]) sc[c][i] = __float_as_uint(-INFINITY);
          }
          // raw scores; the scale (> 0) is applied with the max subtraction.
          // A tree of three-input maxima (depth 4, not a 32-long chain).
          float m[11];
#pragma unroll
          for (int i = 0; i < 10; ++i)
            m[i] = fmax3(__uint_as_float(sc[c][3 * i]), __uint_as_float(sc[c][3 * i + 1]),
                         __uint_as_float(sc[c][3 * i + 2]));
          m[10] = fmaxf(__uint_as_float(sc[c][30]), __uint_as_float(sc[c][31]));
          mx = fmax3(mx, fmax3(fmax3(m[0], m[1], m[2]), fmax3(m[3], m[4], m[5]), fmax3(m[6], m[7], m[8])),
                     fmaxf(m[9], m[10]));
        }
        // the row's maximum over both halves
        xch[h * MT + r] = mx;
        named_bar_sync(pair_bar, 64);
        mx = fmaxf(mx, xch[(h ^ 1) * MT + r]) * qscale;
        PF_TRACE(tq[4] += clock64() - tc; tk = clock64();)
        const float m_new = fmaxf(m_ref[t], mx);
        const bool raise = m_new > m_ref[t] + kRescaleThreshold || (m_ref[t] == -INFINITY && m_new != -INFINITY);
        if (__any_sync(0xffffffffu, raise && m_ref[t] != -INFINITY)) {
          // rare: rescale this half of O's columns (rows that do not raise
          // scale by 1); O is stable, the commit waited for followed PV(j - 1)
          PF_TRACE(const long long tr = clock64();)
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
          PF_TRACE(tq[2] += clock64() - tr;)
        }
        if (raise) m_ref[t] = m_new;
        const float nref = (m_ref[t] == -INFINITY) ? 0.f : -m_ref[t];
        const uint64_t qs2 = f2_pack(qscale, qscale), nr2 = f2_pack(nref, nref);
        // p in pairs (packed fp32x2 arithmetic); row-sum partials in two
        // packed accumulators.  Chunk 2h + c's 32 keys become 16 columns of
        // P pairs (keys 2e, 2e + 1 in column e of the chunk): fp16 P, or the
        // hi pairs of the cache's type with the lo pairs in the 16 columns
        // behind them, so a chunk only overwrites its own, already loaded,
        // scores.
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
        PF_TRACE(tq[6] += clock64() - tk;)
        tmem_wait_st();
        PF_TRACE(tq[3] += clock64() - tc; tc = clock64();)
        tc_fence_before_sync();
        __syncwarp();
        if (lane == 0) mbar_arrive(&bar[P_FULL + t]);
        if (r == 0 && h == 0) PF_TL(5 + t * 2, jj);
        if (lane == 0) PF_TL(8 + warp - kSoftmaxWarp0, jj);
      }
    }
    PF_TRACE(const int slot = (blockIdx.z * gridDim.y + blockIdx.y) * gridDim.x + blockIdx.x;
             if (tid == kSoftmaxWarp0 * 32 && slot < 4096) { for (int i = 0; i < 7; ++i) g_pf_trace[slot][i] = tq[i]; g_pf_trace[slot][7] = clock64() - ts0; })
    // the row sums of both halves (both warps of a pair take part, even
    // after a timeout, so that the pair's named barriers stay matched)
    float lt[NQT];
    bool stored = false;  // TMA stores of output tiles issued by this thread
#pragma unroll
    for (int t = 0; t < NQT; ++t) {
      named_bar_sync(pair_bar, 64);
      xch[h * MT + r] = l[t];
      named_bar_sync(pair_bar, 64);
      lt[t] = l[t] + xch[(h ^ 1) * MT + r];
    }
#pragma unroll
    for (int t = 0; t < NQT; ++t) {
      if (ok && !mbar_wait(&bar[S_FULL + t], n_iter & 1, a.wait_ns)) ok = false;
      if (!ok) break;
      tc_fence_after_sync();
      const int R = t * MT + r;
      const int qi = R / g;
      const bool rv = R < rows_used && qi < nq;
      const uint32_t o_col = C::O_COL + t * D;
      const float inv = lt[t] > 0.f ? vscale / lt[t] : 0.f;
      const int64_t orow_i =
          (static_cast<int64_t>(qs + qt0 + qi) * a.num_q_heads + kvh * g + (R - qi * g)) * a.out_slots + split;
      if (a.otma && (t + 1) * (MT / g) <= nq) {
        // a full tile: this half's columns go through shared memory (the K
        // ring and beyond, free once the tile's last products completed:
        // tile 0's boxes stay inside the K ring, whose last reader, the
        // final QK, precedes tile 0's final commit) as 128-byte-swizzled
        // boxes of 32 columns, then out by TMA stores
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
        named_bar_sync(7 + h, 128);  // the half's four warps wrote their rows
        if ((warp & 3) == 0 && lane == 0) {
          for (int c0 = h * (D / 2); c0 < (h + 1) * (D / 2); c0 += 32)
            tma_store_3d(&a.omap, stage + (c0 / 32) * 16384, c0, kvh * g, qs + qt0 + t * (MT / g));
          bulk_commit_group();
          stored = true;
        }
      } else {
        float *orow = rv ? a.out + orow_i * D : nullptr;
        // this half's columns of the output row
#pragma unroll 1
        for (int c0 = h * (D / 2); c0 < (h + 1) * (D / 2); c0 += 32) {
          float o[32];
          tmem_ld32(trow + o_col + c0, o);
          if (rv) {
#pragma unroll
            for (int i = 0; i < 32; i += 4)
              *reinterpret_cast<float4 *>(orow + c0 + i) =
                  make_float4(o[i] * inv, o[i + 1] * inv, o[i + 2] * inv, o[i + 3] * inv);
          }
        }
      }
      if (rv && h == 0 && a.lse) a.lse[orow_i] = (m_ref[t] + log2f(lt[t])) * kLn2;
    }
    // the stores' shared-memory sources are read before the CTA (or the next
    // tile of a persistent launch) reuses the bytes
    if (stored) bulk_wait_group_read0();
    if (!ok && lane == 0) *s_abort = 1;
  }

  // ---- teardown: after an abort the copies still in flight land first;
  // every product issued for the tile completes before the barriers or the
  // tensor memory are used again
  tc_fence_before_sync();
  __syncthreads();
  if (*s_abort) {
    if (tid == 0) report_error(a.err, a.ws_err, kErrWaitTimeout);
    if (warp == kProducerWarp && lane == 0) {
      if (qtma_tiles != 0 && !a.stall) mbar_wait(&bar[Q_FULL], 0, a.wait_ns);
      for (int t = max(0, *s_last_k - NSK + 1); t <= *s_last_k; ++t)
        mbar_wait(&bar[K_FULL + t % NSK], (t / NSK) & 1, a.wait_ns);
      for (int t = max(0, *s_last_v - NSV + 1); t <= *s_last_v; ++t)
        mbar_wait(&bar[V_FULL + t % NSV], (t / NSV) & 1, a.wait_ns);
    }
  }
  if (warp == kMmaWarp && lane == 0) {
    // a commit after everything this thread issued: its arrival follows the
    // completion of every product (and of the earlier commits' arrivals)
    uint64_t *drain = &bar[P_FULL];
    mbar_init(drain, 1);
    fence_mbar_init();
    umma_commit(drain);
    mbar_wait(drain, 0, a.wait_ns);
  }
  tc_fence_before_sync();
  __syncthreads();
}

// One tile of a grid: query tile bx of gx (counted from the last, so that
// the longest key ranges come first), kv head by, sequence (or sequence x
// key split in prefix mode) bz; all of its KV iterations.
template <int D, int KVT, int PVM, bool NR = false>
__device__ __forceinline__ void prefill_tile(const Args &a, uint8_t *smem, uint32_t tmem, int bx, int by, int bz,
                                             int gx) {
  Seg sg;
  sg.split = a.prefix_mode ? bz % a.num_splits : 0;
  sg.s = a.prefix_mode ? bz / a.num_splits : bz;
  sg.kvh = by;
  sg.qtile = gx - 1 - bx;
  sg.gx = gx;
  sg.it_lo = 0;
  sg.it_hi = -1;
  sg.piece = 0;
  sg.slot = sg.item = sg.c_lo = sg.c_hi = sg.me = 0;
  sg.G = 1;
  sg.item_start = 0;
  sg.U = 1;
  prefill_tile<D, KVT, PVM, NR>(a, smem, tmem, sg);
}

template <int D, int KVT, int PVM>
__global__ void __launch_bounds__(NTHREADS, 1) prefill_tc_kernel(const __grid_constant__ Args a) {
  using C = Cfg<D, KVT, PVM>;
  // launched as a programmatic dependent of the preceding kernel (typically
  // the cache write): nothing is read before its writes are visible
  asm volatile("griddepcontrol.wait;" ::: "memory");
  extern __shared__ uint8_t smem_raw[];
  uint8_t *smem = align1024(smem_raw);
  uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(smem + C::OFF_BAR + NBAR * 8);
  const int warp = threadIdx.x >> 5;
  if (warp == kMmaWarp) tmem_alloc(tmem_slot, C::TMEM_COLS);
  tc_fence_before_sync();
  __syncthreads();
  tc_fence_after_sync();
  const uint32_t tmem = *tmem_slot;
  // grid (kv heads, sequences x splits, query tiles): the CTAs are issued
  // with every item's longest key range first across the whole grid
  prefill_tile<D, KVT, PVM>(a, smem, tmem, blockIdx.z, blockIdx.x, blockIdx.y, gridDim.z);
  tc_fence_before_sync();
  __syncthreads();
  if (warp == kMmaWarp) {
    tc_fence_after_sync();
    tmem_dealloc(tmem, C::TMEM_COLS);
  }
}

template <int D>
inline bool make_map(CUtensorMap *map, const void *base, const pa_kv_desc &d) {
  const bool kv8 = d.kv_dtype == PA_KV_FP8_E4M3 || d.kv_dtype == PA_KV_FP8_E5M2;
  const CUtensorMapDataType dt = kv8                      ? CU_TENSOR_MAP_DATA_TYPE_UINT8
                                 : d.kv_dtype == PA_KV_F16 ? CU_TENSOR_MAP_DATA_TYPE_FLOAT16
                                                           : CU_TENSOR_MAP_DATA_TYPE_BFLOAT16;
  using EncodeTiledFn = CUresult (*)(CUtensorMap *, CUtensorMapDataType, cuuint32_t, void *, const cuuint64_t *,
                                     const cuuint64_t *, const cuuint32_t *, const cuuint32_t *,
                                     CUtensorMapInterleave, CUtensorMapSwizzle, CUtensorMapL2promotion,
                                     CUtensorMapFloatOOBfill);
  static EncodeTiledFn enc = [] {
    void *p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) != cudaSuccess ||
        q != cudaDriverEntryPointSuccess)
      p = nullptr;
    return reinterpret_cast<EncodeTiledFn>(p);
  }();
  if (!enc) return false;
  thread_local MapCache<> cache;  // the last few caches' maps of this thread
  const MapKey key = map_key(base, d.num_blocks, d.num_kv_heads, D, d.kv_dtype);
  if (cache.find(key, map)) return true;
  const cuuint64_t dims[2] = {static_cast<cuuint64_t>(D), static_cast<cuuint64_t>(d.num_blocks) * d.num_kv_heads * 16};
  // 16-bit caches: boxes of 64 columns (128 bytes) x 16 rows; 8-bit caches:
  // a whole row of D bytes (128) x 16 rows
  const cuuint64_t strides[1] = {static_cast<cuuint64_t>(D) * (kv8 ? 1 : 2)};
  const cuuint32_t box[2] = {kv8 ? static_cast<cuuint32_t>(D) : 64u, 16};
  const cuuint32_t estr[2] = {1, 1};
  if (enc(map, dt, 2, const_cast<void *>(base), dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
          CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
          CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
    return false;
  cache.put(key, *map);
  return true;
}

// A step's new K or V rows as a tensor map: [rows][kv heads][D] of the
// cache's 16-bit type, box {64 columns, 1 kv head, 16 rows}: 16 consecutive
// tokens of one kv head land as one 16-row block tile, the layout of a
// cache block's box.  The row extent is the caller's row count, so a box
// that runs past the last row reads zeros.
template <int D>
inline bool make_new_rows_map(CUtensorMap *map, const void *base, int64_t rows, const pa_kv_desc &d) {
  if ((reinterpret_cast<uintptr_t>(base) & 15) != 0 || rows <= 0) return false;
  const CUtensorMapDataType dt =
      d.kv_dtype == PA_KV_F16 ? CU_TENSOR_MAP_DATA_TYPE_FLOAT16 : CU_TENSOR_MAP_DATA_TYPE_BFLOAT16;
  using EncodeTiledFn = CUresult (*)(CUtensorMap *, CUtensorMapDataType, cuuint32_t, void *, const cuuint64_t *,
                                     const cuuint64_t *, const cuuint32_t *, const cuuint32_t *,
                                     CUtensorMapInterleave, CUtensorMapSwizzle, CUtensorMapL2promotion,
                                     CUtensorMapFloatOOBfill);
  static EncodeTiledFn enc = [] {
    void *p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) != cudaSuccess ||
        q != cudaDriverEntryPointSuccess)
      p = nullptr;
    return reinterpret_cast<EncodeTiledFn>(p);
  }();
  if (!enc) return false;
  thread_local MapCache<> cache;
  const MapKey key = map_key(base, rows, d.num_kv_heads, D, d.kv_dtype, -3);
  if (cache.find(key, map)) return true;
  const cuuint64_t dims[3] = {static_cast<cuuint64_t>(D), static_cast<cuuint64_t>(d.num_kv_heads),
                              static_cast<cuuint64_t>(rows)};
  const cuuint64_t strides[2] = {static_cast<cuuint64_t>(D) * 2, static_cast<cuuint64_t>(d.num_kv_heads) * D * 2};
  const cuuint32_t box[3] = {64, 1, 16};
  const cuuint32_t estr[3] = {1, 1, 1};
  if (enc(map, dt, 3, const_cast<void *>(base), dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
          CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
          CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
    return false;
  cache.put(key, *map);
  return true;
}

// The queries' tensor map: [tokens][q heads][D] 16-bit values, box {64
// columns, g heads, 128 / g tokens}, 128-byte swizzle.  The token extent is
// not known on the host (the chunk offsets live on the device); it is set
// to 2^30, and the kernel only asks for boxes of tokens inside a chunk.
// False if the map cannot be made (q not 16-byte aligned, g not dividing
// 128): the threads then stage every Q tile.
template <int D>
inline bool make_qmap(CUtensorMap *map, const void *q, int num_q_heads, int g) {
  if ((reinterpret_cast<uintptr_t>(q) & 15) != 0 || g <= 0 || MT % g != 0) return false;
  using EncodeTiledFn = CUresult (*)(CUtensorMap *, CUtensorMapDataType, cuuint32_t, void *, const cuuint64_t *,
                                     const cuuint64_t *, const cuuint32_t *, const cuuint32_t *,
                                     CUtensorMapInterleave, CUtensorMapSwizzle, CUtensorMapL2promotion,
                                     CUtensorMapFloatOOBfill);
  static EncodeTiledFn enc = [] {
    void *p = nullptr;
    cudaDriverEntryPointQueryResult r;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &r) != cudaSuccess ||
        r != cudaDriverEntryPointSuccess)
      p = nullptr;
    return reinterpret_cast<EncodeTiledFn>(p);
  }();
  if (!enc) return false;
  thread_local MapCache<> cache;
  const MapKey key = map_key(q, num_q_heads, D, g, -1);
  if (cache.find(key, map)) return true;
  const cuuint64_t dims[3] = {static_cast<cuuint64_t>(D), static_cast<cuuint64_t>(num_q_heads), cuuint64_t(1) << 30};
  const cuuint64_t strides[2] = {static_cast<cuuint64_t>(D) * 2, static_cast<cuuint64_t>(num_q_heads) * D * 2};
  const cuuint32_t box[3] = {64, static_cast<cuuint32_t>(g), static_cast<cuuint32_t>(MT / g)};
  const cuuint32_t estr[3] = {1, 1, 1};
  if (enc(map, CU_TENSOR_MAP_DATA_TYPE_UINT16, 3, const_cast<void *>(q), dims, strides, box, estr,
          CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
          CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
    return false;
  cache.put(key, *map);
  return true;
}

// The output's tensor map: [tokens][q heads][D] fp32, box {32 columns, g
// heads, 128 / g tokens}, 128-byte swizzle (the token extent as for q).
// False if it cannot be made (out not 16-byte aligned, g not dividing 128):
// the threads then store every output row themselves.
template <int D>
inline bool make_omap(CUtensorMap *map, const float *out, int num_q_heads, int g) {
  if ((reinterpret_cast<uintptr_t>(out) & 15) != 0 || g <= 0 || MT % g != 0) return false;
  using EncodeTiledFn = CUresult (*)(CUtensorMap *, CUtensorMapDataType, cuuint32_t, void *, const cuuint64_t *,
                                     const cuuint64_t *, const cuuint32_t *, const cuuint32_t *,
                                     CUtensorMapInterleave, CUtensorMapSwizzle, CUtensorMapL2promotion,
                                     CUtensorMapFloatOOBfill);
  static EncodeTiledFn enc = [] {
    void *p = nullptr;
    cudaDriverEntryPointQueryResult r;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &r) != cudaSuccess ||
        r != cudaDriverEntryPointSuccess)
      p = nullptr;
    return reinterpret_cast<EncodeTiledFn>(p);
  }();
  if (!enc) return false;
  thread_local MapCache<> cache;
  const MapKey key = map_key(out, num_q_heads, D, g, -2);
  if (cache.find(key, map)) return true;
  const cuuint64_t dims[3] = {static_cast<cuuint64_t>(D), static_cast<cuuint64_t>(num_q_heads), cuuint64_t(1) << 30};
  const cuuint64_t strides[2] = {static_cast<cuuint64_t>(D) * 4, static_cast<cuuint64_t>(num_q_heads) * D * 4};
  const cuuint32_t box[3] = {32, static_cast<cuuint32_t>(g), static_cast<cuuint32_t>(MT / g)};
  const cuuint32_t estr[3] = {1, 1, 1};
  if (enc(map, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 3, const_cast<float *>(out), dims, strides, box, estr,
          CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_NONE,
          CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
    return false;
  cache.put(key, *map);
  return true;
}

// The kernel's arguments for a call (everything but the grid); false if a
// tensor map of the caches cannot be made.
template <int D>
inline bool make_args(Args *a, const pa_kv_desc &d, float *out, float *lse, const void *q,
                      const int32_t *query_start_loc, const void *k_cache, const void *v_cache,
                      const int32_t *block_tables, int32_t max_blocks_per_seq, const int32_t *context_lens,
                      float scale, bool prefix_mode, int num_splits, int split_len, int out_slots) {
  memset(a, 0, sizeof *a);
  if (!make_map<D>(&a->kmap, k_cache, d) || !make_map<D>(&a->vmap, v_cache, d)) return false;
  a->out = out;
  a->lse = lse;
  a->q = static_cast<const uint16_t *>(q);
  a->query_start_loc = query_start_loc;
  a->block_tables = block_tables;
  a->context_lens = context_lens;
  a->max_blocks_per_seq = max_blocks_per_seq;
  a->num_kv_heads = d.num_kv_heads;
  a->num_q_heads = d.num_q_heads;
  a->g = d.num_q_heads / d.num_kv_heads;
  a->qt = MROWS / a->g;  // queries per CTA
  const bool kv8 = d.kv_dtype == PA_KV_FP8_E4M3 || d.kv_dtype == PA_KV_FP8_E5M2;
  a->qtma = !kv8 && make_qmap<D>(&a->qmap, q, d.num_q_heads, a->g) ? 1 : 0;
  a->otma = !prefix_mode && make_omap<D>(&a->omap, out, d.num_q_heads, a->g) ? 1 : 0;
  a->qscale = scale * ((kv8 && d.k_scale != 0.f) ? d.k_scale : 1.f) * kLog2e;
  a->qscale0 = scale * kLog2e;
  a->vscale = (kv8 && d.v_scale != 0.f) ? d.v_scale : 1.f;
  a->k_scales = kv8 ? d.k_scales : nullptr;
  a->v_scales = kv8 ? d.v_scales : nullptr;
  a->window = d.sliding_window;
  a->chunk = d.attention_chunk;
  a->prefix_mode = prefix_mode ? 1 : 0;
  a->num_splits = prefix_mode ? num_splits : 1;
  a->split_len = split_len;
  a->out_slots = prefix_mode ? out_slots : 1;
  a->err = d.error_word;
  a->checked = d.check_indices;
  a->num_blocks = d.num_blocks;
  const TestHooks hooks = test_hooks();
  a->stall = hooks.stall;
  a->wait_ns = hooks.wait_ns;
  return true;
}

}  // namespace pftc
}  // namespace pa
