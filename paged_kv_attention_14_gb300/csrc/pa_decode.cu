// pa_decode.cu -- host side of pa_decode: kernel choice, launch planning,
// TMA tensor maps, workspace layout and the launch.  The kernels are in
// pa_decode_kernels.cuh (instantiated by pa_decode_simt.cu and
// pa_decode_mma_*.cu).
#include "pa_decode_kernels.cuh"
#include "pa_host_cache.h"

namespace pa {

using dec::KernelInfo;

namespace {

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

int resolve_impl(const pa_kv_desc &d) {
  if (d.decode_impl != PA_DECODE_AUTO) return d.decode_impl;
  return PA_DECODE_MMA;
}

// kv heads handled together by one stage of the MMA kernel (one TMA copy
// moves one block for all of them).  Measured on GB300: bf16 head_dim-128
// tiles are 4 KB per head already and stream best one head per stage; the
// E4M3 kernel (8 consumer warps) is fastest with pairs of heads (2 KB
// tiles), the bf16 head_dim-64 one with groups of 4.
int head_group(const pa_kv_desc &d) {
  const bool b16 = d.kv_dtype == PA_KV_BF16 || d.kv_dtype == PA_KV_F16;
  if (b16 && d.head_dim == 128) return 1;
  if (b16 && d.num_kv_heads % 4 == 0) return 4;
  if (d.num_kv_heads % 2 == 0) return 2;
  return 1;
}

KernelInfo kernel_for(const pa_kv_desc &d, int impl) {
  const int g = d.num_q_heads / d.num_kv_heads;
  if (impl == PA_DECODE_SIMT) return dec::pick_simt(d.head_dim, d.kv_dtype, g);
  const int hg = head_group(d);
  if (d.kv_dtype == PA_KV_BF16) return dec::pick_mma_bf16(d.head_dim, g, hg);
  if (d.kv_dtype == PA_KV_F16) return dec::pick_mma_f16(d.head_dim, g, hg);
  if (d.kv_dtype == PA_KV_FP8_E5M2) return dec::pick_mma_e5m2(d.head_dim, g, hg);
  return dec::pick_mma_fp8(d.head_dim, g, hg);
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

// The cache as TMA sees it.  Rows are (block, kv head, token) triples of
// head_dim elements; one box is the 16 tokens of HG consecutive kv heads of
// one block.  Rows of 256 bytes (bf16, head_dim 128) are cut into two
// 128-byte halves so that the 128-byte swizzle applies: by a third
// dimension (one box per tile) or by two boxes per tile (see kWideMode).
bool encode_cache_map(CUtensorMap *map, const void *base, const pa_kv_desc &d, const KernelInfo &k) {
  EncodeTiledFn enc = encode_tiled();
  if (!enc) return false;
  const bool bf = d.kv_dtype == PA_KV_BF16 || d.kv_dtype == PA_KV_F16;  // 2-byte elements
  const int esz = bf ? 2 : 1;
  const cuuint64_t rowb = static_cast<cuuint64_t>(d.head_dim) * esz;
  const cuuint64_t rows = static_cast<cuuint64_t>(d.num_blocks) * d.num_kv_heads * 16;
  const cuuint32_t box_rows = static_cast<cuuint32_t>(k.hg * 16);
  const CUtensorMapDataType dt = d.kv_dtype == PA_KV_F16 ? CU_TENSOR_MAP_DATA_TYPE_FLOAT16
                                 : bf                      ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16
                                                           : CU_TENSOR_MAP_DATA_TYPE_UINT8;
  const CUtensorMapSwizzle sw = k.swizzle == 128 ? CU_TENSOR_MAP_SWIZZLE_128B : CU_TENSOR_MAP_SWIZZLE_64B;
  const cuuint32_t estr[3] = {1, 1, 1};
  CUresult r;
  if (rowb > 128 && k.wide_mode != dec::kWideTwoBoxes) {
    const cuuint64_t cols = 128 / esz;
    const cuuint64_t halves = rowb / 128;
    const bool half_major = k.wide_mode == dec::kWideHalfMajor;
    const cuuint64_t dims[3] = {cols, half_major ? rows : halves, half_major ? halves : rows};
    const cuuint64_t strides[2] = {half_major ? rowb : 128, half_major ? 128 : rowb};
    const cuuint32_t box[3] = {static_cast<cuuint32_t>(cols), half_major ? box_rows : static_cast<cuuint32_t>(halves),
                               half_major ? static_cast<cuuint32_t>(halves) : box_rows};
    r = enc(map, dt, 3, const_cast<void *>(base), dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE, sw,
            CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  } else {
    const cuuint64_t dims[2] = {static_cast<cuuint64_t>(d.head_dim), rows};
    const cuuint64_t strides[1] = {rowb};
    const cuuint32_t box[2] = {static_cast<cuuint32_t>(rowb > 128 ? 128 / esz : d.head_dim), box_rows};
    r = enc(map, dt, 2, const_cast<void *>(base), dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE, sw,
            CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  }
  return r == CUDA_SUCCESS;
}

// encode_cache_map, remembered per thread for the last few caches
bool make_cache_map(CUtensorMap *map, const void *base, const pa_kv_desc &d, const KernelInfo &k) {
  thread_local MapCache<> cache;
  const MapKey key = map_key(base, d.num_blocks, d.num_kv_heads, d.head_dim, d.kv_dtype, k.hg, k.swizzle, k.wide_mode);
  if (cache.find(key, map)) return true;
  if (!encode_cache_map(map, base, d, k)) return false;
  cache.put(key, *map);
  return true;
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
  const int occ = prepare_kernel(k.fn, k.threads, k.smem);
  if (occ < 1) {
    *why = "the decode kernel does not fit on this device";
    return PA_ERR_CUDA;
  }
  plan->impl = impl;
  plan->slot_heads = k.slot_heads;
  plan->num_groups = d.num_kv_heads / k.hg;
  plan->num_ctas = device_info().sm_count * occ;
  plan->workspace_bytes =
      dec::ws_layout(num_seqs, plan->num_groups, plan->num_ctas, k.slot_heads, d.head_dim).total;
  return PA_OK;
}

namespace dec {

bool make_decode_args(const pa_kv_desc &d, const DecodePlan &plan, float *out, float *lse, const void *q,
                      const void *k_cache, const void *v_cache, const int32_t *block_tables,
                      int32_t max_blocks_per_seq, const int32_t *context_lens, int32_t num_seqs, float scale,
                      void *workspace, DecodeArgs *ap) {
  const KernelInfo k = kernel_for(d, plan.impl);
  const dec::WsLayout w = dec::ws_layout(num_seqs, plan.num_groups, plan.num_ctas, plan.slot_heads, d.head_dim);
  uint8_t *ws = static_cast<uint8_t *>(workspace);
  DecodeArgs &a = *ap;
  memset(&a, 0, sizeof a);
  if (k.mma) {
    if (!make_cache_map(&a.kmap, k_cache, d, k) || !make_cache_map(&a.vmap, v_cache, d, k)) return false;
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
  a.num_groups = plan.num_groups;
  const bool fp8 = d.kv_dtype == PA_KV_FP8_E4M3 || d.kv_dtype == PA_KV_FP8_E5M2;
  const float ks = (fp8 && d.k_scale != 0.f) ? d.k_scale : 1.f;
  a.qscale = scale * ks * dec::kLog2e;
  a.vscale = (fp8 && d.v_scale != 0.f) ? d.v_scale : 1.f;
  a.qscale0 = scale * dec::kLog2e;
  a.k_scales = fp8 ? d.k_scales : nullptr;
  a.v_scales = fp8 ? d.v_scales : nullptr;
  a.window = d.sliding_window;
  a.chunk = d.attention_chunk;
  a.err = reinterpret_cast<int32_t *>(ws);
  a.user_err = d.error_word;
  a.checked = d.check_indices;
  a.num_blocks = d.num_blocks;
  const TestHooks hooks = test_hooks();
  a.stall = hooks.stall;
  a.wait_ns = hooks.wait_ns;
  a.seg_counter = reinterpret_cast<int32_t *>(ws + w.counter_off);
  a.slot_lse = reinterpret_cast<float *>(ws + w.slot_lse_off);
  a.slot_o = reinterpret_cast<float *>(ws + w.slot_o_off);
  return true;
}

}  // namespace dec

cudaError_t launch_decode(const pa_kv_desc &d, const DecodePlan &plan, float *out, float *lse,
                          const void *q, const void *k_cache, const void *v_cache,
                          const int32_t *block_tables, int32_t max_blocks_per_seq,
                          const int32_t *context_lens, int32_t num_seqs, float scale,
                          void *workspace, cudaStream_t stream, const void *k_new, const void *v_new) {
  const KernelInfo k = kernel_for(d, plan.impl);
  dec::DecodeArgs a;
  if (!dec::make_decode_args(d, plan, out, lse, q, k_cache, v_cache, block_tables, max_blocks_per_seq, context_lens,
                             num_seqs, scale, workspace, &a))
    return cudaErrorInvalidValue;
  if (k_new != nullptr) {
    a.k_new = static_cast<const uint8_t *>(k_new);
    a.v_new = static_cast<const uint8_t *>(v_new);
    a.k_write = static_cast<uint8_t *>(const_cast<void *>(k_cache));
    a.v_write = static_cast<uint8_t *>(const_cast<void *>(v_cache));
    a.k_enc = d.k_scale == 0.f ? 1.f : d.k_scale;  // the cache write's per-tensor scales
    a.v_enc = d.v_scale == 0.f ? 1.f : d.v_scale;
  }
  // programmatic dependent launch: the kernel's launch overlaps the tail of
  // the preceding kernel in the stream (typically pa_cache_write); the kernel
  // waits for that kernel's writes before reading anything
  cudaLaunchAttribute pdl[1];
  pdl[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  pdl[0].val.programmaticStreamSerializationAllowed = 1;
  cudaLaunchConfig_t dcfg = {};
  dcfg.gridDim = dim3(plan.num_ctas);
  dcfg.blockDim = dim3(k.threads);
  dcfg.dynamicSmemBytes = k.smem;
  dcfg.stream = stream;
  dcfg.attrs = pdl;
  dcfg.numAttrs = 1;
  void *args[] = {&a};
  return cudaLaunchKernelExC(&dcfg, k.fn, args);
}

}  // namespace pa
