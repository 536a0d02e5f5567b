// pa_merge.cu -- log-sum-exp merge of attention over disjoint key ranges.
//
// Split-KV decoding computes attention over pieces of a sequence's keys and
// recombines them: with M = max_p lse_p and w_p = exp(lse_p - M), the result
// is sum_p w_p o_p / sum_p w_p and its log-sum-exp M + ln sum_p w_p.  The
// pages only name "paged attention" and "chunked prefill" (vllm.cpp
// implementation notes); this identity is what makes a split exact.
//
// One CTA per (sequence, head); each thread owns 4 consecutive output
// elements (float4 loads of every part's row).
#include "pa_device.cuh"
#include "pa_internal.h"

namespace pa {

__global__ void __launch_bounds__(128) merge_kernel(float *__restrict__ out,
                                                     float *__restrict__ lse_out,
                                                     const float *__restrict__ part_o,
                                                     const float *__restrict__ part_lse,
                                                     const int32_t *__restrict__ num_parts,
                                                     int num_heads, int max_parts, int head_dim) {
  const int sh = blockIdx.x;  // s * num_heads + h
  const int s = sh / num_heads;
  const int np = num_parts ? min(__ldg(num_parts + s), max_parts) : max_parts;
  const float *lse_row = part_lse + static_cast<int64_t>(sh) * max_parts;
  constexpr float kLog2e = 1.4426950408889634f;
  float M = -INFINITY;
  for (int p = 0; p < np; ++p) M = fmaxf(M, __ldg(lse_row + p));
  const int d4 = threadIdx.x * 4;
  float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
  float wsum = 0.f;
  if (M != -INFINITY) {
    const float *o_base = part_o + static_cast<int64_t>(sh) * max_parts * head_dim;
    for (int p = 0; p < np; ++p) {
      const float lp = __ldg(lse_row + p);
      if (lp == -INFINITY) continue;
      const float w = exp2f((lp - M) * kLog2e);
      wsum += w;
      if (d4 < head_dim) {
        const float4 o = __ldg(reinterpret_cast<const float4 *>(o_base + static_cast<int64_t>(p) * head_dim + d4));
        acc.x += w * o.x;
        acc.y += w * o.y;
        acc.z += w * o.z;
        acc.w += w * o.w;
      }
    }
  }
  if (d4 < head_dim) {
    const float inv = wsum > 0.f ? 1.f / wsum : 0.f;
    reinterpret_cast<float4 *>(out + static_cast<int64_t>(sh) * head_dim)[threadIdx.x] =
        make_float4(acc.x * inv, acc.y * inv, acc.z * inv, acc.w * inv);
  }
  if (lse_out && threadIdx.x == 0) lse_out[sh] = (M == -INFINITY) ? -INFINITY : M + logf(wsum);
}

cudaError_t launch_merge(float *out, float *lse_out, const float *part_o, const float *part_lse,
                         const int32_t *num_parts, int32_t num_seqs, int32_t num_heads,
                         int32_t max_parts, int32_t head_dim, cudaStream_t stream) {
  const int threads = ((head_dim / 4 + 31) / 32) * 32;
  merge_kernel<<<num_seqs * num_heads, threads, 0, stream>>>(out, lse_out, part_o, part_lse,
                                                             num_parts, num_heads, max_parts,
                                                             head_dim);
  return cudaGetLastError();
}

}  // namespace pa
