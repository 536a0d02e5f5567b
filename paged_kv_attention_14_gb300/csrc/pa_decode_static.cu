// pa_decode_static.cu -- decode attention without a caller-provided workspace.
//
// pa_decode needs a scratch buffer (error word, split-segment records and the
// partial results of sequences split across CTAs) that the caller allocates.
// Some callers cannot allocate device memory at the point where they decode:
// serving loops that run under a fixed device-memory budget and forbid new
// allocations once the KV pool is sized, embedded runtimes whose device
// memory is fully planned at start-up, and plug-ins inside host frameworks
// that own the device allocator and expose no allocation hook to this call
// site.  For them, pa_decode_static runs the same decode kernels on a
// fixed-size scratch array that lives in this library's own device memory.
//
// The array is a file-scope static __device__ buffer of kStaticScratchBytes.
// Every GPU that loads the library holds it until the process exits.  Host
// code cannot use the array's name as a device address, so on the first call
// on each device (with that device current) the address is looked up once
// with cudaGetSymbolAddress and cached.
#include <mutex>

#include "pa.h"
#include "pa_internal.h"

namespace {

// Maximum scratch of one call.  The decode workspace is a few hundred KB for
// typical batches (it grows with the number of persistent CTAs, the query
// heads per kv head group and the number of sequences); calls needing more
// are rejected with PA_ERR_WORKSPACE.
constexpr size_t kStaticScratchBytes = size_t(8) << 20;

static __device__ __align__(256) unsigned char g_static_scratch[kStaticScratchBytes];

constexpr int kMaxDevices = 64;
std::mutex g_scratch_mutex;
void *g_scratch_ptr[kMaxDevices] = {};

pa_status static_fail(pa_status st, const char *msg) {
  pa::set_last_error(msg);
  return st;
}

// Device address of the scratch array on the current device; looked up once
// per device.
cudaError_t scratch_address(void **out) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev < 0 || dev >= kMaxDevices) return cudaErrorInvalidDevice;
  std::lock_guard<std::mutex> lock(g_scratch_mutex);
  if (!g_scratch_ptr[dev]) {
    void *p = nullptr;
    e = cudaGetSymbolAddress(&p, g_static_scratch);
    if (e != cudaSuccess) return e;
    g_scratch_ptr[dev] = p;
  }
  *out = g_scratch_ptr[dev];
  return cudaSuccess;
}

}  // namespace

extern "C" {

PA_API pa_status pa_decode_static(const pa_kv_desc *desc, float *out, float *lse, const void *q,
                                  const void *k_cache, const void *v_cache, const int32_t *block_tables,
                                  int32_t max_blocks_per_seq, const int32_t *context_lens, int32_t num_seqs,
                                  int32_t max_context_len, float scale, pa_stream_t stream) {
  // every argument check of pa_decode first, so that a call that fails on
  // its arguments enqueues nothing
  pa::DecodePlan plan;
  const pa_status st = pa::validate_decode(desc, out, lse, q, k_cache, v_cache, block_tables, max_blocks_per_seq,
                                           context_lens, num_seqs, max_context_len, scale, &plan);
  if (st != PA_OK) return st;
  if (num_seqs == 0) {
    pa::set_last_error("");
    return PA_OK;
  }
  if (plan.workspace_bytes > kStaticScratchBytes)
    return static_fail(PA_ERR_WORKSPACE,
                       "this batch needs more decode scratch than the 8 MiB static array; use pa_decode");
  void *scratch = nullptr;
  cudaError_t e = scratch_address(&scratch);
  if (e != cudaSuccess) return static_fail(PA_ERR_CUDA, cudaGetErrorString(e));
  // The array keeps the previous call's contents: its error word and merge
  // counters (the first 256 bytes plus one int32 per sequence and kv head)
  // must start at zero, the rest is rewritten by every launch.
  const size_t head = 256 + sizeof(int32_t) * static_cast<size_t>(num_seqs) * desc->num_kv_heads;
  const cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  e = cudaMemsetAsync(scratch, 0, head < plan.workspace_bytes ? head : plan.workspace_bytes, s);
  if (e != cudaSuccess) return static_fail(PA_ERR_CUDA, cudaGetErrorString(e));
  e = pa::launch_decode(*desc, plan, out, lse, q, k_cache, v_cache, block_tables, max_blocks_per_seq, context_lens,
                        num_seqs, scale, scratch, s);
  if (e != cudaSuccess) return static_fail(PA_ERR_CUDA, cudaGetErrorString(e));
  pa::set_last_error("");
  return PA_OK;
}

}  // extern "C"
