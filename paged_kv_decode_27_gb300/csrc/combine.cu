// combine.cu -- log-sum-exp merge of the split-K partials of paged decode.
//
// Partition p of a sequence leaves its normalised output o_p[d] and
// lse_p = log2 sum_i 2^(x_i) over its tokens (scores x in the log2 domain).
// With M = max_p lse_p and w_p = 2^(lse_p - M):
//     out[d] = sum_p w_p o_p[d] / sum_p w_p,
// which equals the softmax over the whole context exactly (up to fp32
// rounding).  One warp per (sequence, query head); sequences that fit in one
// partition were written directly by the decode kernel and are skipped.
#include "pa_common.cuh"
#include "pa_internal.h"

namespace pa {

template <typename T, int D>
__global__ void __launch_bounds__(128) combine_kernel(const DecodeArgs a) {
  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const long long pair = static_cast<long long>(blockIdx.x) * 4 + warp;
  if (pair >= static_cast<long long>(a.num_seqs) * a.num_q_heads) return;
  const int s = static_cast<int>(pair / a.num_q_heads);

  int ctx = __ldg(a.context_lens + s);
  const int cap = min(a.max_blocks_per_seq * kBlock, a.max_context_len);
  ctx = ctx < 0 ? 0 : (ctx > cap ? cap : ctx);
  const int nblk = (ctx + kBlock - 1) / kBlock;
  const int n = (nblk + a.part_blocks - 1) / a.part_blocks;
  if (n <= 1) return;

  const float* lse = a.ws_lse + pair * a.max_splits;
  const float* po = a.ws_o + pair * a.max_splits * D;
  float M = -INFINITY;
  for (int p = lane; p < n; p += 32) M = fmaxf(M, lse[p]);
  M = warp_max_xor(M, 1, 16);
  float L = 0.f;
  if (M != -INFINITY)
    for (int p = lane; p < n; p += 32) L += exp2f(lse[p] - M);
  L = warp_sum_xor(L, 1, 16);
  const float inv = (L > 0.f) ? 1.f / L : 0.f;

  T* out = static_cast<T*>(a.out) + pair * D;
  for (int d = lane; d < D; d += 32) {
    float o = 0.f;
    if (M != -INFINITY) {
      for (int p = 0; p < n; ++p) {
        const float lp = lse[p];
        if (lp != -INFINITY) o = fmaf(exp2f(lp - M), po[static_cast<size_t>(p) * D + d], o);
      }
    }
    out[d] = Elem<T>::from_f(o * inv);
  }
}

namespace {
template <typename T, int D>
cudaError_t launch_combine_t(const DecodeArgs& a, cudaStream_t stream) {
  const long long pairs = static_cast<long long>(a.num_seqs) * a.num_q_heads;
  const long long blocks = (pairs + 3) / 4;
  combine_kernel<T, D><<<static_cast<unsigned>(blocks), 128, 0, stream>>>(a);
  return cudaGetLastError();
}
}  // namespace

cudaError_t launch_combine(const DecodeArgs& a, int dtype, cudaStream_t stream) {
  switch (dtype) {
    case PA_F32:
      return a.head_dim == 128 ? launch_combine_t<float, 128>(a, stream)
                               : launch_combine_t<float, 64>(a, stream);
    case PA_BF16:
      return a.head_dim == 128 ? launch_combine_t<__nv_bfloat16, 128>(a, stream)
                               : launch_combine_t<__nv_bfloat16, 64>(a, stream);
    default:
      return a.head_dim == 128 ? launch_combine_t<__half, 128>(a, stream)
                               : launch_combine_t<__half, 64>(a, stream);
  }
}

}  // namespace pa
