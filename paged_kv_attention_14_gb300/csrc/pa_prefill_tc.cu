// pa_prefill_tc.cu -- causal chunked-prefill attention on the 5th-generation
// tensor cores (tcgen05.mma, accumulators in tensor memory), bf16 KV.
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
//    the other tile.  Q is staged once; K/V are walked in 64-key tiles
//    gathered block by block through the block table by TMA (two
//    128-byte-swizzled boxes per 16-token block) into two 3-stage rings, one
//    for K and one for V, shared by both Q tiles.  A K slot is released as
//    soon as the QKs that read it complete, a V slot after its PVs, so the
//    copies run up to three tiles ahead of the tensor cores.
//  * Warp 9 (one thread) issues the MMAs: S_t = Q_t K^T (M 128, N 64, K 16 x
//    head_dim/16) into one of tile t's two TMEM S buffers, and O_t += P_t V
//    (M 128, N head_dim, K 16 x 4) with P_t from shared memory and V read
//    MN-major, in the order QK_A(j+1), QK_B(j+1), PV_A(j), PV_B(j): the
//    scores of the next KV tile are computed while the softmax of this one
//    runs.
//  * Warps 0-3 (tile A) and 4-7 (tile B), one thread per row with the row's
//    64 scores in registers, do the online softmax: scale, causal mask, row
//    max, exp2, row sum, and write P
//    as a bf16 hi + lo pair (P = hi + lo to ~2^-17 relative; two PV MMAs)
//    so the bf16 tensor-core result keeps near-fp32 accuracy.  The running
//    max is only raised (and O rescaled in TMEM) when it grows by more than
//    2^8, so O is rarely touched before the end.
//  * Keys past the chunk's last position are masked; V rows past it are
//    zeroed in shared memory before the last PV (0 * NaN would not vanish).
//  * Warp 8 issues the TMA copies and prefetches block-table entries one
//    tile ahead.
//  * Every wait is bounded; on a timeout the kernel records an error bit,
//    lets its own MMAs and copies drain and frees its TMEM before returning.
#include <cuda.h>
#include <string.h>

#include "pa_device.cuh"
#include "pa_internal.h"

namespace pa {
namespace pftc {

constexpr float kLog2e = 1.4426950408889634f;
constexpr float kLn2 = 0.6931471805599453f;
constexpr int KT = 64;         // keys per KV tile
constexpr int MT = 128;        // rows of one Q tile (one TMEM lane per row)
constexpr int NQT = 2;         // Q tiles per CTA (ping-pong between two softmax warpgroups)
constexpr int MROWS = MT * NQT;
constexpr int NTHREADS = 320;  // warps 0-3 softmax A, 4-7 softmax B, 8 TMA producer, 9 MMA issuer
constexpr int kProducerWarp = 8;
constexpr int kMmaWarp = 9;
constexpr int NST = 3;         // stages of the K ring and of the V ring
constexpr float kRescaleThreshold = 8.f;  // log2 units

struct Args {
  CUtensorMap kmap;  // cache as [rows = blocks * kv heads * 16][D], box {64, 16}
  CUtensorMap vmap;
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
  float qscale;
};

// Error bits of the prefill kernel (a bounded wait ran out); device code
// sets them, nothing else uses them.
static __device__ int g_prefill_err;

// Optional timeline counters (compiled only with -DPA_PREFILL_TRACE), per
// CTA slot (blockIdx linearised, first 4096): softmax warp 0 lane 0 cycles
// [0] waiting for S, [1] loading S from TMEM, [2] masking and max, [3]
// waiting for the previous PV, [4] rescaling O, [5] exp2 and P stores, [6]
// fence and arrive, [7] total; MMA thread cycles [8] waiting for K/V, [9]
// waiting for S_FREE, [10] waiting for P, [11] total; producer [12] waiting
// for a free K/V buffer, [13] total; [14] KV tiles.
#ifdef PA_PREFILL_TRACE
static __device__ unsigned long long g_pf_trace[4096][16];
#define PF_TRACE(...) __VA_ARGS__
#else
#define PF_TRACE(...)
#endif

template <int D>
struct Cfg {
  static constexpr int HALVES = D / 64;          // 128-byte column halves of a row
  static constexpr int QHALF = MT * 128;         // bytes of one half of one Q tile
  static constexpr int QB = HALVES * QHALF;      // one Q tile
  static constexpr int KVHALF = KT * 128;        // bytes of one half of a K or V tile
  static constexpr int KVB = HALVES * KVHALF;
  static constexpr int PB = MT * KT * 2;         // one P matrix (hi or lo), 128 x 64 bf16
  static constexpr int OFF_Q = 0;                // [NQT]
  static constexpr int OFF_K = OFF_Q + NQT * QB;    // [NST]
  static constexpr int OFF_V = OFF_K + NST * KVB;   // [NST]
  static constexpr int OFF_P = OFF_V + NST * KVB;   // [NQT][hi, lo]
  static constexpr int OFF_BAR = OFF_P + NQT * 2 * PB;
  static constexpr int SMEM = OFF_BAR + 256 + 1024;  // + barriers, TMEM slot, 1024-B alignment slack
  static_assert(SMEM <= 232448, "shared memory of one CTA");
  // TMEM columns: two S buffers of each Q tile (KT each), then O of each Q
  // tile (D each)
  static constexpr uint32_t S_COL = 0;
  static constexpr uint32_t O_COL = NQT * 2 * KT;
  static constexpr uint32_t COLS_USED = NQT * 2 * KT + NQT * D;
  static constexpr uint32_t TMEM_COLS = COLS_USED <= 256 ? 256 : 512;
  static constexpr uint32_t IDESC_QK = umma_idesc_bf16(MT, KT, false, false);
  static constexpr uint32_t IDESC_PV = umma_idesc_bf16(MT, D, false, true);
  // bytes landed per 16-token block of K (or of V), all halves
  static constexpr uint32_t BLOCK_BYTES = HALVES * 16u * 128u;
};

// barriers: K_FULL[NST], K_EMPTY[NST], V_FULL[NST], V_EMPTY[NST],
// S_FULL[tile][2], S_FREE[tile][2], P_FULL[tile], PV_DONE[tile]
enum Bar {
  K_FULL = 0,
  K_EMPTY = K_FULL + NST,
  V_FULL = K_EMPTY + NST,
  V_EMPTY = V_FULL + NST,
  S_FULL = V_EMPTY + NST,
  S_FREE = S_FULL + 4,
  P_FULL = S_FREE + 4,
  PV_DONE = P_FULL + 2,
  NBAR = PV_DONE + 2
};
static_assert(NBAR * 8 + 16 <= 256, "barriers, TMEM slot and flags fit their 256 bytes");

template <int D>
__global__ void __launch_bounds__(NTHREADS, 1) prefill_tc_kernel(const __grid_constant__ Args a) {
  using C = Cfg<D>;
  // launched as a programmatic dependent of the preceding kernel (typically
  // the cache write): nothing is read before its writes are visible
  asm volatile("griddepcontrol.wait;" ::: "memory");
  extern __shared__ uint8_t smem_raw[];
  uint8_t *smem = reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint64_t *bar = reinterpret_cast<uint64_t *>(smem + C::OFF_BAR);
  uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(bar + NBAR);
  int *s_abort = reinterpret_cast<int *>(tmem_slot + 1);
  int *s_last_k = s_abort + 1;  // last KV tile whose K copies the producer issued
  int *s_last_v = s_abort + 2;  // ... and whose V copies

  const int s = blockIdx.z;
  const int kvh = blockIdx.y;
  const int qtile = gridDim.x - 1 - blockIdx.x;  // longest key ranges first
  const int qs = __ldg(a.query_start_loc + s);
  const int q_len = __ldg(a.query_start_loc + s + 1) - qs;
  const int qt0 = qtile * a.qt;
  if (qt0 >= q_len) return;
  const int L = __ldg(a.context_lens + s);
  const int nq = min(a.qt, q_len - qt0);
  const int base_pos = L - q_len + qt0;  // position of query qt0
  const int kv_end = base_pos + nq;      // keys [0, kv_end) are needed
  const int n_tiles = (kv_end + KT - 1) / KT;
  const int tid = threadIdx.x;
  const int warp = tid >> 5;
  const int lane = tid & 31;
  const int g = a.g;
  const int rows_used = a.qt * g;

  if (tid == 0) {
    for (int i = 0; i < NST; ++i) {
      mbar_init(&bar[K_FULL + i], 1);
      mbar_init(&bar[K_EMPTY + i], 1);
      mbar_init(&bar[V_FULL + i], 1);
      mbar_init(&bar[V_EMPTY + i], 1);
    }
    for (int i = 0; i < 2; ++i) {
      mbar_init(&bar[P_FULL + i], 4);
      mbar_init(&bar[PV_DONE + i], 1);
    }
    for (int i = 0; i < 4; ++i) {
      mbar_init(&bar[S_FULL + i], 1);
      mbar_init(&bar[S_FREE + i], 4);
    }
    *s_abort = 0;
    *s_last_k = -1;
    *s_last_v = -1;
    fence_mbar_init();
  }
  if (warp == kMmaWarp) tmem_alloc(tmem_slot, C::TMEM_COLS);

  // ---- Q tiles: row R = query * g + head (tile R / 128, lane R % 128),
  // [tile][half][row][128 B], 128-B swizzle
  {
    constexpr int CHUNKS = D / 8;  // 16-byte chunks per row
    for (int i = tid; i < MROWS * CHUNKS; i += NTHREADS) {
      const int R = i / CHUNKS;
      const int ch = i - R * CHUNKS;
      const int qi = R / g;
      const bool ok = R < rows_used && qi < nq;
      const uint16_t *src = a.q;
      if (ok) src = a.q + (static_cast<int64_t>(qs + qt0 + qi) * a.num_q_heads + kvh * g + (R - qi * g)) * D + ch * 8;
      const int r = R & (MT - 1);
      uint8_t *dst = smem + C::OFF_Q + (R / MT) * C::QB + (ch >> 3) * C::QHALF + r * 128 + (((ch & 7) ^ (r & 7)) << 4);
      cp_async16(dst, src, ok);
    }
    cp_async_commit();
    cp_async_wait<0>();
    fence_proxy_async_smem();
  }
  tc_fence_before_sync();
  __syncthreads();
  tc_fence_after_sync();
  const uint32_t tmem = *tmem_slot;
  const uint32_t sbase = smem_u32(smem);

  if (warp == kProducerWarp) {
    // ------------------------------------------------------ TMA producer
    const int32_t *table = a.block_tables + static_cast<int64_t>(s) * a.max_blocks_per_seq;
    const uint64_t pol = l2_evict_first_policy();
    // lane -> (K or V, block of the tile, half)
    const int kv = lane / (4 * C::HALVES);
    const int bi = (lane / C::HALVES) & 3;
    const int hh = lane % C::HALVES;
    const bool issuer = lane < 2 * 4 * C::HALVES;
    int phys_next = 0;
    if (issuer && bi * 16 < kv_end) phys_next = __ldg(table + bi);
    PF_TRACE(const long long tp0 = clock64(); long long tp_wait = 0;)
    for (int j = 0; j < n_tiles; ++j) {
      const int st = j % NST;
      const uint32_t ph = (j / NST) & 1;
      const int phys = phys_next;
      const int key0 = j * KT;
      const int lb = (j + 1) * 4 + bi;  // prefetch the next tile's block id
      phys_next = (issuer && lb * 16 < kv_end) ? __ldg(table + lb) : 0;
      const int nblk = min(4, (kv_end - key0 + 15) / 16);
      const int row = (phys * a.num_kv_heads + kvh) * 16;
      // K of tile j (its slot frees once the QKs of tile j - NST completed),
      // then V of tile j (once the PVs of tile j - NST completed)
      bool ok = true;
#pragma unroll 1
      for (int part = 0; part < 2 && ok; ++part) {
        const int full = (part ? V_FULL : K_FULL) + st;
        PF_TRACE(const long long tw = clock64();)
        if (!mbar_wait(&bar[(part ? V_EMPTY : K_EMPTY) + st], ph ^ 1)) {
          ok = false;
          break;
        }
        PF_TRACE(tp_wait += clock64() - tw;)
        if (lane == 0) mbar_arrive_expect_tx(&bar[full], nblk * C::BLOCK_BYTES);
        __syncwarp();
        if (issuer && kv == part && bi < nblk) {
          uint8_t *dst = smem + (part ? C::OFF_V : C::OFF_K) + st * C::KVB + hh * C::KVHALF + bi * 16 * 128;
          tma_load_2d(dst, part ? &a.vmap : &a.kmap, hh * 64, row, &bar[full], pol);
        }
        if (lane == 0) *(part ? s_last_v : s_last_k) = j;
      }
      if (!ok) {
        if (lane == 0) *s_abort = 1;
        break;
      }
    }
    PF_TRACE(const int slot = (blockIdx.z * gridDim.y + blockIdx.y) * gridDim.x + blockIdx.x;
             if (lane == 0 && slot < 4096) { g_pf_trace[slot][12] = tp_wait; g_pf_trace[slot][13] = clock64() - tp0; g_pf_trace[slot][14] = n_tiles; })
  } else if (warp == kMmaWarp) {
    // --------------------------------------------------------- MMA issuer
    if (lane == 0) {
      bool ok = true;
      auto qk = [&](int t, int j) {  // S_t[j & 1] = Q_t K_j^T
        const int b = j & 1;
        const uint32_t qbase = sbase + C::OFF_Q + t * C::QB;
        const uint32_t kbase = sbase + C::OFF_K + (j % NST) * C::KVB;
#pragma unroll
        for (int kk = 0; kk < D / 16; ++kk) {
          const uint64_t ad = umma_desc_sw128(qbase + (kk >> 2) * C::QHALF + (kk & 3) * 32, 16, 1024);
          const uint64_t bd = umma_desc_sw128(kbase + (kk >> 2) * C::KVHALF + (kk & 3) * 32, 16, 1024);
          umma_bf16_ss(tmem + C::S_COL + (t * 2 + b) * KT, ad, bd, C::IDESC_QK, kk > 0 ? 1u : 0u);
        }
        umma_commit(&bar[S_FULL + t * 2 + b]);
      };
      auto pv = [&](int t, int j) {  // O_t += P_t V_j
        const uint32_t pbase = sbase + C::OFF_P + t * 2 * C::PB;
        const uint32_t vbase = sbase + C::OFF_V + (j % NST) * C::KVB;
#pragma unroll
        for (int part = 0; part < 2; ++part) {  // hi, then lo
#pragma unroll
          for (int kk = 0; kk < KT / 16; ++kk) {
            const uint64_t ad = umma_desc_sw128(pbase + part * C::PB + kk * 32, 16, 1024);
            const uint64_t bd = umma_desc_sw128(vbase + kk * 2048, C::KVHALF, 1024);
            umma_bf16_ss(tmem + C::O_COL + t * D, ad, bd, C::IDESC_PV, (j > 0 || part > 0 || kk > 0) ? 1u : 0u);
          }
        }
        umma_commit(&bar[PV_DONE + t]);
      };
      // S of KV tile j + 1 is computed before the PV of tile j, so the next
      // scores are ready when a tile's softmax finishes
      PF_TRACE(const long long tm0 = clock64(); long long tm_kv = 0, tm_sf = 0, tm_p = 0; long long tw;)
      if (!mbar_wait(&bar[K_FULL], 0)) ok = false;
      if (ok) {
        tc_fence_after_sync();
        for (int t = 0; t < NQT; ++t) qk(t, 0);
        umma_commit(&bar[K_EMPTY]);
      }
      for (int j = 0; j < n_tiles && ok; ++j) {
        if (j + 1 < n_tiles) {
          const int j1 = j + 1;
          PF_TRACE(tw = clock64();)
          if (!mbar_wait(&bar[K_FULL + j1 % NST], (j1 / NST) & 1)) {
            ok = false;
            break;
          }
          PF_TRACE(tm_kv += clock64() - tw;)
          for (int t = 0; t < NQT && ok; ++t) {
            PF_TRACE(tw = clock64();)
            if (!mbar_wait(&bar[S_FREE + t * 2 + (j1 & 1)], ((j1 >> 1) & 1) ^ 1)) {
              ok = false;
              break;
            }
            PF_TRACE(tm_sf += clock64() - tw;)
            tc_fence_after_sync();
            qk(t, j1);
          }
          if (ok) umma_commit(&bar[K_EMPTY + j1 % NST]);  // K of tile j + 1 is consumed
        }
        if (!ok) break;
        PF_TRACE(tw = clock64();)
        if (!mbar_wait(&bar[V_FULL + j % NST], (j / NST) & 1)) {
          ok = false;
          break;
        }
        PF_TRACE(tm_kv += clock64() - tw;)
        for (int t = 0; t < NQT && ok; ++t) {
          PF_TRACE(tw = clock64();)
          if (!mbar_wait(&bar[P_FULL + t], j & 1)) {
            ok = false;
            break;
          }
          PF_TRACE(tm_p += clock64() - tw;)
          tc_fence_after_sync();
          pv(t, j);
        }
        if (ok) umma_commit(&bar[V_EMPTY + j % NST]);  // both tiles are done with V of tile j
      }
      if (!ok) *s_abort = 1;
      PF_TRACE(const int slot = (blockIdx.z * gridDim.y + blockIdx.y) * gridDim.x + blockIdx.x;
               if (slot < 4096) { g_pf_trace[slot][8] = tm_kv; g_pf_trace[slot][9] = tm_sf; g_pf_trace[slot][10] = tm_p; g_pf_trace[slot][11] = clock64() - tm0; })
    }
    __syncwarp();
  } else {
    // ------------------------------------------------ softmax, one row per thread
    const int t = warp >> 2;  // Q tile of this warpgroup
    const int r = tid & (MT - 1);
    const int R = t * MT + r;
    // TMEM lane = row; warp w reads lanes 32 (w % 4) .. 32 (w % 4) + 31
    const uint32_t trow = tmem + (static_cast<uint32_t>((warp & 3) * 32) << 16);
    const uint32_t o_col = C::O_COL + t * D;
    const int qi = R / g;
    const bool rv = R < rows_used && qi < nq;
    const int pos = rv ? base_pos + qi : -1;  // keys <= pos are visible
    const float qscale = a.qscale;
    float m_ref = -INFINITY, l = 0.f;
    bool ok = true;
    PF_TRACE(const long long ts0 = clock64(); long long tq[7] = {0, 0, 0, 0, 0, 0, 0}; long long tc;)
    for (int j = 0; j < n_tiles; ++j) {
      const int sb = j & 1;
      PF_TRACE(tc = clock64();)
      if (!mbar_wait(&bar[S_FULL + t * 2 + sb], (j >> 1) & 1)) {
        ok = false;
        break;
      }
      PF_TRACE(tq[0] += clock64() - tc; tc = clock64();)
      tc_fence_after_sync();
      float sv[KT];
      const uint32_t s_col = C::S_COL + (t * 2 + sb) * KT;
      tmem_ld32(trow + s_col, *reinterpret_cast<float(*)[32]>(&sv[0]));
      tmem_ld32(trow + s_col + 32, *reinterpret_cast<float(*)[32]>(&sv[32]));
      tc_fence_before_sync();
      __syncwarp();
      if (lane == 0) mbar_arrive(&bar[S_FREE + t * 2 + sb]);
      PF_TRACE(tq[1] += clock64() - tc; tc = clock64();)
      const int key0 = j * KT;
      // raw scores; the scale (> 0) is applied with the max subtraction
      float mx = -INFINITY;
      if (key0 + KT - 1 <= pos) {
#pragma unroll
        for (int c = 0; c < KT; ++c) mx = fmaxf(mx, sv[c]);
      } else {
#pragma unroll
        for (int c = 0; c < KT; ++c) {
          sv[c] = (key0 + c <= pos) ? sv[c] : -INFINITY;
          mx = fmaxf(mx, sv[c]);
        }
      }
      mx *= qscale;
      if (t == 0 && j == n_tiles - 1 && kv_end - key0 < KT) {
        // V rows past the last needed key: zero (stale or poisoned data),
        // after this tile's V copies landed; tile 0's PV of this KV tile is
        // issued before tile 1's
        if (!mbar_wait(&bar[V_FULL + j % NST], (j / NST) & 1)) {
          ok = false;
          break;
        }
        const int kval = kv_end - key0;
        for (int i = r; i < (KT - kval) * C::HALVES * 8; i += MT) {
          const int row = kval + i / (C::HALVES * 8);
          const int rem = i % (C::HALVES * 8);
          *reinterpret_cast<uint4 *>(smem + C::OFF_V + (j % NST) * C::KVB + (rem >> 3) * C::KVHALF + row * 128 +
                                     (rem & 7) * 16) = make_uint4(0, 0, 0, 0);
        }
      }
      PF_TRACE(tq[2] += clock64() - tc; tc = clock64();)
      // this tile's P buffer and O are free once its previous PV completed
      if (j > 0) {
        if (!mbar_wait(&bar[PV_DONE + t], (j - 1) & 1)) {
          ok = false;
          break;
        }
        tc_fence_after_sync();
      }
      PF_TRACE(tq[3] += clock64() - tc; tc = clock64();)
      const float m_new = fmaxf(m_ref, mx);
      const bool raise = m_new > m_ref + kRescaleThreshold || (m_ref == -INFINITY && m_new != -INFINITY);
      if (__any_sync(0xffffffffu, raise && m_ref != -INFINITY)) {
        // rescale this warp's O rows in TMEM (rows that do not raise scale by 1)
        const float corr = (raise && m_ref != -INFINITY) ? exp2f(m_ref - m_new) : 1.f;
        if (raise) l *= corr;
#pragma unroll 1
        for (int c0 = 0; c0 < D; c0 += 32) {
          float o[32];
          tmem_ld32(trow + o_col + c0, o);
#pragma unroll
          for (int i = 0; i < 32; ++i) o[i] *= corr;
          tmem_st32(trow + o_col + c0, o);
        }
      }
      if (raise) m_ref = m_new;
      PF_TRACE(tq[4] += clock64() - tc; tc = clock64();)
      const float nref = (m_ref == -INFINITY) ? 0.f : -m_ref;
      uint8_t *ph_ = smem + C::OFF_P + t * 2 * C::PB + r * 128;
      uint8_t *pl_ = ph_ + C::PB;
#pragma unroll
      for (int c8 = 0; c8 < KT / 8; ++c8) {
        uint32_t hi[4], lo[4];
#pragma unroll
        for (int e = 0; e < 4; ++e) {
          const float p0 = ex2_approx(fmaf(sv[c8 * 8 + 2 * e], qscale, nref));
          const float p1 = ex2_approx(fmaf(sv[c8 * 8 + 2 * e + 1], qscale, nref));
          l += p0 + p1;
          hi[e] = pack_bf16x2(p0, p1);
          lo[e] = pack_bf16x2(p0 - bf16lo(hi[e]), p1 - bf16hi(hi[e]));
        }
        const int off = ((c8 ^ (r & 7)) << 4);
        *reinterpret_cast<uint4 *>(ph_ + off) = make_uint4(hi[0], hi[1], hi[2], hi[3]);
        *reinterpret_cast<uint4 *>(pl_ + off) = make_uint4(lo[0], lo[1], lo[2], lo[3]);
      }
      PF_TRACE(tq[5] += clock64() - tc; tc = clock64();)
      fence_proxy_async_smem();
      tc_fence_before_sync();
      __syncwarp();
      if (lane == 0) mbar_arrive(&bar[P_FULL + t]);
      PF_TRACE(tq[6] += clock64() - tc;)
    }
    PF_TRACE(const int slot = (blockIdx.z * gridDim.y + blockIdx.y) * gridDim.x + blockIdx.x;
             if (tid == 0 && slot < 4096) { for (int i = 0; i < 7; ++i) g_pf_trace[slot][i] = tq[i]; g_pf_trace[slot][7] = clock64() - ts0; })
    if (ok && !mbar_wait(&bar[PV_DONE + t], (n_tiles - 1) & 1)) ok = false;
    if (ok) {
      tc_fence_after_sync();
      const float inv = l > 0.f ? 1.f / l : 0.f;
      float *orow = nullptr;
      if (rv) orow = a.out + (static_cast<int64_t>(qs + qt0 + qi) * a.num_q_heads + kvh * g + (R - qi * g)) * D;
#pragma unroll 1
      for (int c0 = 0; c0 < D; c0 += 32) {
        float o[32];
        tmem_ld32(trow + o_col + c0, o);
        if (rv) {
#pragma unroll
          for (int i = 0; i < 32; i += 4)
            *reinterpret_cast<float4 *>(orow + c0 + i) = make_float4(o[i] * inv, o[i + 1] * inv, o[i + 2] * inv, o[i + 3] * inv);
        }
      }
      if (rv && a.lse)
        a.lse[static_cast<int64_t>(qs + qt0 + qi) * a.num_q_heads + kvh * g + (R - qi * g)] = (m_ref + log2f(l)) * kLn2;
    } else if (lane == 0) {
      *s_abort = 1;
    }
  }

  // ---- teardown: drain on abort, free TMEM
  tc_fence_before_sync();
  __syncthreads();
  if (*s_abort) {
    if (tid == 0) atomicOr(&g_prefill_err, kErrWaitTimeout);
    if (warp == kProducerWarp && lane == 0) {
      // the copies of the last NST issued tiles must land before exit
      for (int t = max(0, *s_last_k - NST + 1); t <= *s_last_k; ++t) mbar_wait(&bar[K_FULL + t % NST], (t / NST) & 1);
      for (int t = max(0, *s_last_v - NST + 1); t <= *s_last_v; ++t) mbar_wait(&bar[V_FULL + t % NST], (t / NST) & 1);
    }
    if (warp == kMmaWarp && lane == 0) {
      // wait (bounded) for every MMA this thread issued before freeing TMEM
      uint64_t *drain = &bar[S_FULL];
      mbar_init(drain, 1);
      fence_mbar_init();
      umma_commit(drain);
      mbar_wait(drain, 0);
    }
    __syncthreads();
  }
  if (warp == kMmaWarp) {
    tc_fence_after_sync();
    tmem_dealloc(tmem, C::TMEM_COLS);
  }
}

template <int D>
bool make_map(CUtensorMap *map, const void *base, const pa_kv_desc &d) {
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
  const cuuint64_t dims[2] = {static_cast<cuuint64_t>(D), static_cast<cuuint64_t>(d.num_blocks) * d.num_kv_heads * 16};
  const cuuint64_t strides[1] = {static_cast<cuuint64_t>(D) * 2};
  const cuuint32_t box[2] = {64, 16};
  const cuuint32_t estr[2] = {1, 1};
  return enc(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void *>(base), dims, strides, box, estr,
             CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
             CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

template <int D>
cudaError_t launch(const pa_kv_desc &d, float *out, float *lse, const void *q, const int32_t *query_start_loc,
                   const void *k_cache, const void *v_cache, const int32_t *block_tables, int32_t max_blocks_per_seq,
                   const int32_t *context_lens, int32_t num_seqs, int32_t max_q_len, float scale,
                   cudaStream_t stream) {
  Args a;
  memset(&a, 0, sizeof a);
  if (!make_map<D>(&a.kmap, k_cache, d) || !make_map<D>(&a.vmap, v_cache, d)) return cudaErrorInvalidValue;
  a.out = out;
  a.lse = lse;
  a.q = static_cast<const uint16_t *>(q);
  a.query_start_loc = query_start_loc;
  a.block_tables = block_tables;
  a.context_lens = context_lens;
  a.max_blocks_per_seq = max_blocks_per_seq;
  a.num_kv_heads = d.num_kv_heads;
  a.num_q_heads = d.num_q_heads;
  a.g = d.num_q_heads / d.num_kv_heads;
  a.qt = MROWS / a.g;  // queries per CTA
  a.qscale = scale * kLog2e;
  const int qtiles = (max_q_len + a.qt - 1) / a.qt;
  if (qtiles == 0 || num_seqs == 0) return cudaSuccess;
  auto fn = &prefill_tc_kernel<D>;
  cudaError_t e = cudaFuncSetAttribute(fn, cudaFuncAttributeMaxDynamicSharedMemorySize, Cfg<D>::SMEM);
  if (e != cudaSuccess) return e;
  cudaLaunchAttribute pdl[1];
  pdl[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  pdl[0].val.programmaticStreamSerializationAllowed = 1;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(qtiles, d.num_kv_heads, num_seqs);
  cfg.blockDim = dim3(NTHREADS);
  cfg.dynamicSmemBytes = Cfg<D>::SMEM;
  cfg.stream = stream;
  cfg.attrs = pdl;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, fn, a);
}

}  // namespace pftc

#ifdef PA_PREFILL_TRACE
extern "C" PA_API int pa_debug_prefill_trace_read(unsigned long long *host, int rows) {
  if (rows > 4096) rows = 4096;
  return static_cast<int>(cudaMemcpyFromSymbol(host, pftc::g_pf_trace, sizeof(unsigned long long) * 16 * rows));
}
#endif

cudaError_t launch_prefill_tc(const pa_kv_desc &d, float *out, float *lse, const void *q,
                              const int32_t *query_start_loc, const void *k_cache, const void *v_cache,
                              const int32_t *block_tables, int32_t max_blocks_per_seq, const int32_t *context_lens,
                              int32_t num_seqs, int32_t max_q_len, float scale, cudaStream_t stream) {
  if (d.head_dim == 128)
    return pftc::launch<128>(d, out, lse, q, query_start_loc, k_cache, v_cache, block_tables, max_blocks_per_seq,
                             context_lens, num_seqs, max_q_len, scale, stream);
  return pftc::launch<64>(d, out, lse, q, query_start_loc, k_cache, v_cache, block_tables, max_blocks_per_seq,
                          context_lens, num_seqs, max_q_len, scale, stream);
}

}  // namespace pa
