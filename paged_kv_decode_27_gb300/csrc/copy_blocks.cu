// copy_blocks.cu -- whole-block copies for copy-on-write in the paged pool.
//
// When a sequence appends into a last block that another sequence's table
// also holds, the block manager hands out a fresh block and the pair
// (source, destination); this kernel copies every KV head of the source block
// into the destination, for K and V, before the new tokens are written.  One
// thread per 16 bytes; a pair's block is H_kv * 16 * D * elem bytes.
#include "pa_common.cuh"
#include "pa_internal.h"

namespace pa {

__global__ void __launch_bounds__(256)
copy_blocks_kernel(uint4* __restrict__ k_pool, uint4* __restrict__ v_pool, const int32_t* __restrict__ pairs,
                   int num_pairs, int chunks_per_block, int num_blocks, int* status) {
  grid_dependency_wait();
  const long long idx = static_cast<long long>(blockIdx.x) * blockDim.x + threadIdx.x;
  if (idx >= static_cast<long long>(num_pairs) * chunks_per_block) return;
  const int pr = static_cast<int>(idx / chunks_per_block);
  const int c = static_cast<int>(idx - static_cast<long long>(pr) * chunks_per_block);
  const int src = __ldg(pairs + 2 * pr);
  const int dst = __ldg(pairs + 2 * pr + 1);
  if (src < 0 || src >= num_blocks || dst < 0 || dst >= num_blocks) {
    if (c == 0 && blockIdx.y == 0) flag_status(status, PA_DEV_BAD_BLOCK_ID);
    return;
  }
  uint4* pool = blockIdx.y == 0 ? k_pool : v_pool;
  pool[static_cast<size_t>(dst) * chunks_per_block + c] = pool[static_cast<size_t>(src) * chunks_per_block + c];
}

cudaError_t launch_copy_blocks(void* k_pool, void* v_pool, const int32_t* pairs, int num_pairs, int block_bytes,
                               int num_blocks, int* status, cudaStream_t stream) {
  if (num_pairs == 0) return cudaSuccess;
  const int cpb = block_bytes / 16;
  const long long n = static_cast<long long>(num_pairs) * cpb;
  const long long blocks = (n + 255) / 256;
  if (blocks > 0x7fffffffLL) return cudaErrorInvalidValue;
  copy_blocks_kernel<<<dim3(static_cast<unsigned>(blocks), 2), 256, 0, stream>>>(
      static_cast<uint4*>(k_pool), static_cast<uint4*>(v_pool), pairs, num_pairs, cpb, num_blocks, status);
  return cudaGetLastError();
}

}  // namespace pa
