// append_kv.cu -- scatter each step's new K/V rows into the 16-token block pool.
//
// The per-step KV write of an inference engine ("Mini inference engine (KV
// cache + sampling + quantization)", step 2: append on each step; "LLM
// Inference Server", Stage 1: new K/V written in place into pre-allocated
// buffers), routed through a slot mapping (slot = block*16 + offset) into the
// paged pool of "LLM Inference Server", Paged KV-Cache Block Allocator.
//
// A pure indexed copy: every thread moves one 16-byte chunk of one (token,
// head) row of K or V, so reads of k_new/v_new and writes into the pool are
// both 128-bit and coalesced along the row.  Bit-exact by construction.
#include "pa_common.cuh"
#include "pa_internal.h"

namespace pa {

__global__ void __launch_bounds__(256)
append_kv_kernel(uint4* __restrict__ k_pool, uint4* __restrict__ v_pool,
                 const int64_t* __restrict__ slot_mapping, const uint4* __restrict__ k_new,
                 const uint4* __restrict__ v_new, int num_tokens, int num_kv_heads,
                 int chunks_per_row, int num_blocks, int* status) {
  allow_dependents();   // the decode/prefill that follows waits for our writes itself
  const long long idx = static_cast<long long>(blockIdx.x) * blockDim.x + threadIdx.x;
  const long long per_tensor = static_cast<long long>(num_tokens) * num_kv_heads * chunks_per_row;
  if (idx >= per_tensor) return;
  const bool is_v = blockIdx.y != 0;
  const int c = static_cast<int>(idx % chunks_per_row);
  const long long th = idx / chunks_per_row;
  const int h = static_cast<int>(th % num_kv_heads);
  const long long t = th / num_kv_heads;

  const long long slot = __ldg(slot_mapping + t);
  if (slot < 0) return;                                   // padding token
  if (slot >= static_cast<long long>(num_blocks) * kBlock) {
    if (c == 0 && h == 0 && !is_v) flag_status(status, PA_DEV_BAD_SLOT);
    return;
  }
  const long long blk = slot / kBlock;
  const int off = static_cast<int>(slot % kBlock);
  const size_t dst = ((static_cast<size_t>(blk) * num_kv_heads + h) * kBlock + off) *
                         static_cast<size_t>(chunks_per_row) + c;
  const size_t src = static_cast<size_t>(th) * chunks_per_row + c;
  if (is_v) {
    v_pool[dst] = __ldcs(v_new + src);
  } else {
    k_pool[dst] = __ldcs(k_new + src);
  }
}

cudaError_t launch_append(void* k_pool, void* v_pool, const int64_t* slot_mapping,
                          const void* k_new, const void* v_new, int num_tokens,
                          int num_kv_heads, int row_bytes, int num_blocks, int* status,
                          cudaStream_t stream) {
  if (num_tokens == 0) return cudaSuccess;
  const int cpr = row_bytes / 16;
  const long long per_tensor = static_cast<long long>(num_tokens) * num_kv_heads * cpr;
  const int threads = 256;
  const long long blocks = (per_tensor + threads - 1) / threads;
  if (blocks > 0x7fffffffLL) return cudaErrorInvalidValue;
  dim3 grid(static_cast<unsigned>(blocks), 2);
  append_kv_kernel<<<grid, threads, 0, stream>>>(
      static_cast<uint4*>(k_pool), static_cast<uint4*>(v_pool), slot_mapping,
      static_cast<const uint4*>(k_new), static_cast<const uint4*>(v_new), num_tokens,
      num_kv_heads, cpr, num_blocks, status);
  return cudaGetLastError();
}

}  // namespace pa
