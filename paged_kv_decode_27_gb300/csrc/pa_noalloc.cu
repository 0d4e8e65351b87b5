// pa_noalloc.cu -- split-K decode attention for callers that cannot allocate.
//
// pa_decode_attention needs a caller-provided device workspace for the
// split-K partials whenever a sequence spans more than one partition.  Some
// callers cannot provide one: a serving loop that must not call cudaMalloc
// once it is running (a fixed memory budget whose pool may not grow), an
// embedder that hands this library only the tensors it already owns, or a
// plain C host with no device allocator of its own.
// pa_decode_attention_noalloc serves them: the partials go to the file-scope
// device array below instead of a caller buffer.  The first call
// that needs the array on a device looks up its address there; make that
// first call before any stream capture.  Calls that overlap on the GPU (on
// different streams of one device) share the array and race.
//
// The array is PA_NOALLOC_SCRATCH_BYTES (32 MiB) per device.  It is part of
// the library's module, so every GPU that loads the library holds it until the
// process exits.  Only the split-K completion counters at its start must be
// zero when a call begins; each call clears the ones it uses.  The partials
// the merge reads are written earlier by the same call.
#include <cstdio>
#include <mutex>

#include "pa.h"
#include "pa_internal.h"

// Split-K partials of pa_decode_attention_noalloc (shared by every call on a device).
static __device__ __align__(256) unsigned char g_pa_noalloc_scratch[PA_NOALLOC_SCRATCH_BYTES];

namespace {

// Device address of the array for the current device.  Looked up once per
// device, with that device current, on the first call that needs it: in host
// code the array's name is only a host-side stand-in, so the real address must
// come from cudaGetSymbolAddress.  The address is kept together with the
// context it was found in; after a device reset (a new context, whose module
// may sit elsewhere) the next call looks it up again.
void* noalloc_scratch(cudaError_t* err) {
  static std::mutex mu;
  static void* addr[64] = {};
  static void* addr_ctx[64] = {};
  int dev = 0;
  *err = cudaGetDevice(&dev);
  if (*err != cudaSuccess) return nullptr;
  if (dev < 0 || dev >= 64) {
    *err = cudaErrorInvalidDevice;
    return nullptr;
  }
  std::lock_guard<std::mutex> lock(mu);
  if (!addr[dev] || addr_ctx[dev] != pa::current_context()) {
    void* p = nullptr;
    *err = cudaGetSymbolAddress(&p, g_pa_noalloc_scratch);
    if (*err != cudaSuccess) return nullptr;
    addr[dev] = p;
    addr_ctx[dev] = pa::current_context();
  }
  return addr[dev];
}

}  // namespace

extern "C" PA_API int pa_decode_attention_noalloc(void* out, const void* q, const void* k_pool,
                                                  const void* v_pool, const int32_t* block_tables,
                                                  const int32_t* context_lens, float scale, int num_seqs,
                                                  int num_q_heads, int max_blocks_per_seq, int max_context_len,
                                                  int partition_size, const pa_pool_desc* pool, void* stream) {
  // Pure host arithmetic first: a shape whose partials do not fit is refused
  // before anything touches the device.
  const size_t need =
      pa_decode_workspace_size(num_seqs, num_q_heads, max_context_len, partition_size, pool);
  if (need > static_cast<size_t>(PA_NOALLOC_SCRATCH_BYTES)) {
    char msg[320];
    snprintf(msg, sizeof(msg),
             "pa_decode_attention_noalloc: this batch needs %zu bytes of split-K scratch but the "
             "built-in array holds %zu bytes; pass a larger partition_size or call "
             "pa_decode_attention with a workspace",
             need, static_cast<size_t>(PA_NOALLOC_SCRATCH_BYTES));
    return pa::set_last_error(PA_ERR_INVALID, msg);
  }
  void* ws = nullptr;
  size_t ws_bytes = 0;
  if (need > 0) {
    cudaError_t e = cudaSuccess;
    ws = noalloc_scratch(&e);
    if (!ws) {
      char msg[200];
      snprintf(msg, sizeof(msg), "pa_decode_attention_noalloc: scratch address lookup failed: %s",
               cudaGetErrorString(e));
      return pa::set_last_error(PA_ERR_CUDA, msg);
    }
    ws_bytes = PA_NOALLOC_SCRATCH_BYTES;
    // The split-K completion counters at the start of the array must be zero
    // when the kernel starts; clear the ones this call uses (no allocation).
    // (batches beyond the 65536-entry counter region are refused by
    // pa_decode_attention below, so nothing is enqueued for them)
    const long long pairs = static_cast<long long>(num_seqs) * pool->num_kv_heads;
    if (pairs <= 65536)
      e = cudaMemsetAsync(ws, 0, static_cast<size_t>(pairs) * sizeof(int), static_cast<cudaStream_t>(stream));
    if (e != cudaSuccess) {
      char msg[200];
      snprintf(msg, sizeof(msg), "pa_decode_attention_noalloc: clearing the counters failed: %s",
               cudaGetErrorString(e));
      return pa::set_last_error(PA_ERR_CUDA, msg);
    }
  }
  // Every other check, and the launches, are those of pa_decode_attention.
  return pa_decode_attention(out, q, k_pool, v_pool, block_tables, context_lens, scale, num_seqs,
                             num_q_heads, max_blocks_per_seq, max_context_len, partition_size, pool, ws,
                             ws_bytes, stream);
}
