// decode_simt.cu -- paged decode attention on the CUDA cores (the fp32 path).
//
// Same work split as the tensor-core kernel -- grid (split, KV head, sequence),
// W warps taking the partition's blocks round-robin, a shared-memory merge of
// the warp states -- but each warp walks its blocks token by token with lanes
// spread over the head dimension: coalesced loads of the K and V rows (a
// group of tokens at a time, so a block waits on a few load latencies, not
// one per token), one warp-shuffle reduction per query head for the score,
// and an fp32 online softmax update.  Used for fp32 pools, where tensor-core precision would not
// meet the 1e-5 bar.
#include "decode_merge.cuh"
#include "pa_common.cuh"
#include "pa_internal.h"

namespace pa {

template <typename T, int N>
__device__ __forceinline__ void load_row_f(const T* p, float* o) {
  constexpr int B = N * static_cast<int>(sizeof(T));
  if constexpr (B == 16) {
    const uint4 u = __ldg(reinterpret_cast<const uint4*>(p));
    const T* e = reinterpret_cast<const T*>(&u);
#pragma unroll
    for (int i = 0; i < N; ++i) o[i] = Elem<T>::to_f(e[i]);
  } else if constexpr (B == 8) {
    const uint2 u = __ldg(reinterpret_cast<const uint2*>(p));
    const T* e = reinterpret_cast<const T*>(&u);
#pragma unroll
    for (int i = 0; i < N; ++i) o[i] = Elem<T>::to_f(e[i]);
  } else if constexpr (B == 4) {
    const uint32_t u = __ldg(reinterpret_cast<const unsigned int*>(p));
    const T* e = reinterpret_cast<const T*>(&u);
#pragma unroll
    for (int i = 0; i < N; ++i) o[i] = Elem<T>::to_f(e[i]);
  } else {
#pragma unroll
    for (int i = 0; i < N; ++i) o[i] = Elem<T>::to_f(p[i]);
  }
}

template <typename T, int D, int W>
__global__ void __launch_bounds__(W * 32) decode_simt_kernel(const DecodeArgs a) {
  constexpr int DPL = D / 32;   // head-dim elements per lane
  __shared__ float red_o[W * 8 * D];
  __shared__ float red_m[W * 8];
  __shared__ float red_l[W * 8];

  const int split = blockIdx.x;
  const int kvh = blockIdx.y;
  const int s = blockIdx.z;
  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const int G = a.num_q_heads / a.num_kv_heads;

  grid_dependency_wait();   // inputs may come from the kernel just before us
  const int ctx = checked_context(a, s, threadIdx.x == 0 && split == 0 && kvh == 0);
  const int nblk_seq = (ctx + kBlock - 1) / kBlock;
  const int n_splits = (nblk_seq + a.part_blocks - 1) / a.part_blocks;
  if (ctx == 0) {
    if (split == 0) store_zero_rows<T, D>(a, G, s, kvh, W * 32);
    return;
  }
  if (split >= n_splits) return;
  if (a.k_new != nullptr && split == n_splits - 1) {   // decode step with the append fused in
    write_step_token<T, D>(a, s, kvh, ctx, W * 32);
    __syncthreads();
  }
  const int blk0 = split * a.part_blocks;
  const int nblk = min(a.part_blocks, nblk_seq - blk0);

  const T* kpool = static_cast<const T*>(a.k_pool);
  const T* vpool = static_cast<const T*>(a.v_pool);
  float qv[8][DPL];
#pragma unroll
  for (int h = 0; h < 8; ++h) {
    if (h < G) {
      load_row_f<T, DPL>(static_cast<const T*>(a.q) +
                             (static_cast<size_t>(s) * a.num_q_heads + kvh * G + h) * D + lane * DPL,
                         qv[h]);
    } else {
#pragma unroll
      for (int e = 0; e < DPL; ++e) qv[h][e] = 0.f;
    }
  }
  float m[8], l[8], acc[8][DPL];
#pragma unroll
  for (int h = 0; h < 8; ++h) {
    m[h] = -INFINITY;
    l[h] = 0.f;
#pragma unroll
    for (int e = 0; e < DPL; ++e) acc[h][e] = 0.f;
  }

  for (int j = warp; j < nblk; j += W) {
    const int lb = blk0 + j;
    const int id = __ldg(a.block_tables + static_cast<size_t>(s) * a.max_blocks_per_seq + lb);
    if (id < 0 || id >= a.num_blocks) {
      if (lane == 0) flag_status(a.status, PA_DEV_BAD_BLOCK_ID);
      continue;
    }
    const int nvalid = min(kBlock, ctx - lb * kBlock);
    const size_t tile = (static_cast<size_t>(id) * a.num_kv_heads + kvh) * kBlock * D;
    // TB tokens' K and V rows are loaded together (32 registers a lane), so a
    // block costs kBlock / TB memory latencies instead of one per token; rows
    // past the context lie inside the block's tile and are loaded but unused
    constexpr int TB = 16 / DPL;
    static_assert(kBlock % TB == 0, "token groups tile the block");
    for (int t0 = 0; t0 < nvalid; t0 += TB) {
      float kr[TB][DPL], vr[TB][DPL];
#pragma unroll
      for (int u = 0; u < TB; ++u) {
        load_row_f<T, DPL>(kpool + tile + static_cast<size_t>(t0 + u) * D + lane * DPL, kr[u]);
        load_row_f<T, DPL>(vpool + tile + static_cast<size_t>(t0 + u) * D + lane * DPL, vr[u]);
      }
#pragma unroll
      for (int u = 0; u < TB; ++u) {
        if (t0 + u >= nvalid) break;
#pragma unroll
        for (int h = 0; h < 8; ++h) {
          if (h < G) {
            float x = 0.f;
#pragma unroll
            for (int e = 0; e < DPL; ++e) x = fmaf(qv[h][e], kr[u][e], x);
            x = warp_sum_xor(x, 1, 16) * a.scale_log2;
            const float mn = fmaxf(m[h], x);
            const float al = exp2f(m[h] - mn);
            const float p = exp2f(x - mn);
            l[h] = l[h] * al + p;
#pragma unroll
            for (int e = 0; e < DPL; ++e) acc[h][e] = fmaf(acc[h][e], al, p * vr[u][e]);
            m[h] = mn;
          }
        }
      }
    }
  }

#pragma unroll
  for (int h = 0; h < 8; ++h) {
    if (h < G) {
#pragma unroll
      for (int e = 0; e < DPL; ++e) red_o[(warp * 8 + h) * D + lane * DPL + e] = acc[h][e];
      if (lane == 0) {
        red_m[warp * 8 + h] = m[h];
        red_l[warp * 8 + h] = l[h];
      }
    }
  }
  __syncthreads();
  cta_merge_store<T, W, D>(a, red_o, red_m, red_l, G, s, kvh, split, n_splits);
}

namespace {
template <typename T, int D>
cudaError_t launch_simt_t(const DecodeArgs& a, cudaStream_t stream) {
  constexpr int W = 4;
  dim3 grid(a.max_splits, a.num_kv_heads, a.num_seqs);
  return launch_pdl(decode_simt_kernel<T, D, W>, grid, dim3(W * 32), 0, stream, a);
}
}  // namespace

cudaError_t launch_decode_simt(const DecodeArgs& a, int dtype, cudaStream_t stream) {
  switch (dtype) {
    case PA_F32:
      return a.head_dim == 128 ? launch_simt_t<float, 128>(a, stream) : launch_simt_t<float, 64>(a, stream);
    case PA_BF16:
      return a.head_dim == 128 ? launch_simt_t<__nv_bfloat16, 128>(a, stream)
                               : launch_simt_t<__nv_bfloat16, 64>(a, stream);
    default:
      return a.head_dim == 128 ? launch_simt_t<__half, 128>(a, stream) : launch_simt_t<__half, 64>(a, stream);
  }
}

}  // namespace pa
