// copy_blocks.cu -- whole-block copies for copy-on-write in the paged pool.
//
// When a sequence appends into a last block that another sequence's table
// also holds, the block manager hands out a fresh block and the pair
// (source, destination); this kernel copies every KV head of the source block
// into the destination, for K and V (and, for an INT8 cache, the matching
// rows of the K and V scale arrays), before the new tokens are written.  One
// thread per 16 bytes; grid.y picks the array.  A pair's block is
// H_kv * 16 * D * elem bytes of a pool and H_kv * 16 * 4 bytes of a scale
// array.
#include "pa_common.cuh"
#include "pa_internal.h"

namespace pa {

__global__ void __launch_bounds__(256)
copy_blocks_kernel(const CopyArrays arrs, const int32_t* __restrict__ pairs, int num_pairs, int num_blocks,
                   int* status) {
  grid_dependency_wait();
  const int which = blockIdx.y;
  const int cpb = arrs.chunks_per_block[which];
  const long long idx = static_cast<long long>(blockIdx.x) * blockDim.x + threadIdx.x;
  if (idx >= static_cast<long long>(num_pairs) * cpb) return;
  const int pr = static_cast<int>(idx / cpb);
  const int c = static_cast<int>(idx - static_cast<long long>(pr) * cpb);
  const int src = __ldg(pairs + 2 * pr);
  const int dst = __ldg(pairs + 2 * pr + 1);
  if (src < 0 || src >= num_blocks || dst < 0 || dst >= num_blocks) {
    if (c == 0 && which == 0) flag_status(status, PA_DEV_BAD_BLOCK_ID);
    return;
  }
  uint4* a = static_cast<uint4*>(arrs.ptr[which]);
  a[static_cast<size_t>(dst) * cpb + c] = a[static_cast<size_t>(src) * cpb + c];
}

cudaError_t launch_copy_blocks(const CopyArrays& arrs, int num_arrays, const int32_t* pairs, int num_pairs,
                               int num_blocks, int* status, cudaStream_t stream) {
  if (num_pairs == 0) return cudaSuccess;
  int cpb_max = 0;
  for (int i = 0; i < num_arrays; ++i) cpb_max = arrs.chunks_per_block[i] > cpb_max ? arrs.chunks_per_block[i] : cpb_max;
  const long long n = static_cast<long long>(num_pairs) * cpb_max;
  const long long blocks = (n + 255) / 256;
  if (blocks > 0x7fffffffLL) return cudaErrorInvalidValue;
  copy_blocks_kernel<<<dim3(static_cast<unsigned>(blocks), num_arrays), 256, 0, stream>>>(arrs, pairs, num_pairs,
                                                                                         num_blocks, status);
  return cudaGetLastError();
}

}  // namespace pa
