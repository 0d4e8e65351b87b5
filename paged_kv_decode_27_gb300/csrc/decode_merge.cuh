// decode_merge.cuh -- merge the per-warp online-softmax states of one CTA and
// store either the final output (single partition) or one split-K partial;
// for split-K, the CTA that finishes last for its (sequence, KV head) then
// merges all partials (the log-sum-exp combine, fused into the decode kernel).
//
// A CTA works on one (sequence, KV head) and its query columns: the G query
// heads of the group at each of the a.q_len query positions (q_len = 1 for
// decode), column c = i * G + h for position i and head h.  Each warp leaves,
// for every column c < G * q_len (stride NC per warp):
//   red_m[w][c]  reference of the log2-domain scores (the running maximum, or
//                a lazily raised value below it),
//   red_l[w][c]  sum of 2^(x - m) over the warp's tokens,
//   red_o[w][c][d] sum of 2^(x - m) * v[d].
// A warp that saw no token has m = -inf, l = 0, o = 0 and weighs nothing.
#pragma once

#include "pa_common.cuh"
#include "pa_internal.h"

namespace pa {

// Row of q / out (and, times max_splits, of the split-K partials) that holds
// query column c of (sequence s, KV head kvh): q and out are
// [num_seqs][q_len][num_q_heads][D].
__device__ __forceinline__ size_t query_row(const DecodeArgs& a, int s, int kvh, int G, int c) {
  const int i = c / G;
  const int h = c - i * G;
  return (static_cast<size_t>(s) * a.q_len + i) * a.num_q_heads + kvh * G + h;
}

// Four consecutive outputs of one row, rounded once to T and stored together
// (8 bytes for bf16/fp16, 16 for fp32; rows start 16-byte aligned).
template <typename T>
__device__ __forceinline__ void store_out4(T* dst, float4 v) {
  if constexpr (sizeof(T) == 4) {
    *reinterpret_cast<float4*>(dst) = v;
  } else {
    T t[4] = {Elem<T>::from_f(v.x), Elem<T>::from_f(v.y), Elem<T>::from_f(v.z), Elem<T>::from_f(v.w)};
    *reinterpret_cast<uint2*>(dst) = *reinterpret_cast<const uint2*>(t);
  }
}

// Log-sum-exp merge of the n_parts split-K partials of (sequence s, KV head
// kvh) into the output rows: with M = max_p lse_p and w_p = 2^(lse_p - M),
// out = sum_p w_p o_p / sum_p w_p -- the softmax over the whole context.
// Threads tid = 0 .. nthreads-1 share the G * q_len * D / 4 groups of four
// consecutive outputs; each thread keeps the loads of kBatch partials (their
// lse and a float4 of their output) in flight together, so a merge of up to
// kBatch partitions costs about one L2 round trip per group it owns.
template <typename T, int D>
__device__ __forceinline__ void merge_split_partials(const DecodeArgs& a, int s, int kvh, int G, int n_parts,
                                                     int tid, int nthreads) {
  T* out = static_cast<T*>(a.out);
  const int ncols = G * a.q_len;
  constexpr int V4 = D / 4;       // float4 groups per row
  constexpr int kBatch = 16;      // partials whose loads are in flight together
  for (int idx = tid; idx < ncols * V4; idx += nthreads) {
    const int c = idx / V4;
    const int d4 = idx - c * V4;
    const size_t qr = query_row(a, s, kvh, G, c);
    const size_t row0 = qr * a.max_splits;
    // a running max over batches of partitions
    float M = -INFINITY, L = 0.f;
    float4 O = make_float4(0.f, 0.f, 0.f, 0.f);
    for (int p0 = 0; p0 < n_parts; p0 += kBatch) {
      float lp[kBatch];
      float4 op[kBatch];
#pragma unroll
      for (int k = 0; k < kBatch; ++k) {
        const bool in = p0 + k < n_parts;
        lp[k] = in ? __ldcg(a.ws_lse + row0 + p0 + k) : -INFINITY;
        op[k] = in ? __ldcg(reinterpret_cast<const float4*>(a.ws_o + (row0 + p0 + k) * D) + d4)
                   : make_float4(0.f, 0.f, 0.f, 0.f);
      }
      float mb = M;
#pragma unroll
      for (int k = 0; k < kBatch; ++k) mb = fmaxf(mb, lp[k]);
      if (mb == -INFINITY) continue;
      const float r = exp2f(M - mb);      // 0 while M is still -inf
      L *= r;
      O.x *= r;
      O.y *= r;
      O.z *= r;
      O.w *= r;
#pragma unroll
      for (int k = 0; k < kBatch; ++k) {
        const float w = exp2f(lp[k] - mb);   // 0 for empty partitions
        L += w;
        O.x = fmaf(w, op[k].x, O.x);
        O.y = fmaf(w, op[k].y, O.y);
        O.z = fmaf(w, op[k].z, O.z);
        O.w = fmaf(w, op[k].w, O.w);
      }
      M = mb;
    }
    const float4 o = L > 0.f ? make_float4(O.x / L, O.y / L, O.z / L, O.w / L) : make_float4(0.f, 0.f, 0.f, 0.f);
    store_out4<T>(out + qr * D + 4 * d4, o);
  }
}

template <typename T, int W, int D, int NC = 8, int NTHREADS = W * 32>
__device__ __forceinline__ void cta_merge_store(const DecodeArgs& a, const float* red_o,
                                                const float* red_m, const float* red_l, int G,
                                                int s, int kvh, int split, int n_splits) {
  __shared__ int s_last;
  const int ncols = G * a.q_len;
  for (int idx = threadIdx.x; idx < ncols * D; idx += NTHREADS) {
    const int c = idx / D;
    const int d = idx - c * D;
    float M = -INFINITY;
#pragma unroll
    for (int w = 0; w < W; ++w) M = fmaxf(M, red_m[w * NC + c]);
    float L = 0.f, O = 0.f;
    if (M != -INFINITY) {
#pragma unroll
      for (int w = 0; w < W; ++w) {
        const float mw = red_m[w * NC + c];
        const float f = (mw == -INFINITY) ? 0.f : exp2f(mw - M);
        L += f * red_l[w * NC + c];
        O += f * red_o[(w * NC + c) * D + d];
      }
    }
    const size_t qr = query_row(a, s, kvh, G, c);
    const float o = (L > 0.f) ? O / L : 0.f;
    if (n_splits == 1) {
      T* out = static_cast<T*>(a.out);
      out[qr * D + d] = Elem<T>::from_f(o);
    } else {
      const size_t row = qr * a.max_splits + split;
      a.ws_o[row * D + d] = o;
      if (d == 0) a.ws_lse[row] = (L > 0.f) ? M + log2f(L) : -INFINITY;
    }
  }
  if (n_splits == 1) return;

  // ---- split-K: the last CTA of this (sequence, KV head) merges every
  // partition by log-sum-exp.  With M = max_p lse_p and w_p = 2^(lse_p - M),
  // out = sum_p w_p o_p / sum_p w_p -- the softmax over the whole context.
  // Release/acquire: the CTA barrier orders every thread's partial stores
  // before thread 0's acq_rel atomic; the last CTA's atomic acquires the other
  // partitions' stores, and the second barrier passes that on to its threads.
  __syncthreads();
  int* counter = a.ws_count + static_cast<size_t>(s) * a.num_kv_heads + kvh;
  if (threadIdx.x == 0) {
    int prev;
    asm volatile("atom.add.acq_rel.gpu.global.s32 %0, [%1], 1;" : "=r"(prev) : "l"(counter) : "memory");
    s_last = (prev == n_splits - 1);
  }
  __syncthreads();
  if (!s_last) return;
  merge_split_partials<T, D>(a, s, kvh, G, n_splits, threadIdx.x, NTHREADS);
  // leave the counter at zero for the next call on this workspace
  if (threadIdx.x == 0) *counter = 0;
}

// A sequence with an empty context produces zero rows for its query columns.
template <typename T, int D>
__device__ __forceinline__ void store_zero_rows(const DecodeArgs& a, int G, int s, int kvh,
                                                int nthreads) {
  T* out = static_cast<T*>(a.out);
  for (int idx = threadIdx.x; idx < G * a.q_len * D; idx += nthreads) {
    const int c = idx / D;
    const int d = idx - c * D;
    out[query_row(a, s, kvh, G, c) * D + d] = Elem<T>::from_f(0.f);
  }
}

// Append fused into a decode step: the CTA that holds a sequence's last
// partition writes the step's new token (position ctx - 1) of its KV head
// into the pool, K and V, 16 bytes per thread.  The caller orders the write
// before its own reads of that block (a CTA barrier, plus a generic-to-async
// proxy fence when the reads are TMA copies).
template <typename T, int D>
__device__ __forceinline__ void write_step_token(const DecodeArgs& a, int s, int kvh, int ctx, int nthreads) {
  constexpr int CH = D * static_cast<int>(sizeof(T)) / 16;   // 16-byte chunks per row
  const int pos = ctx - 1;
  const int id = __ldg(a.block_tables + static_cast<size_t>(s) * a.max_blocks_per_seq + pos / kBlock);
  if (id < 0 || id >= a.num_blocks) {
    if (threadIdx.x == 0) flag_status(a.status, PA_DEV_BAD_BLOCK_ID);
    return;
  }
  const size_t row = (static_cast<size_t>(id) * a.num_kv_heads + kvh) * kBlock + pos % kBlock;
  const size_t src = static_cast<size_t>(s) * a.num_kv_heads + kvh;
  for (int c = threadIdx.x; c < 2 * CH; c += nthreads) {
    const bool is_v = c >= CH;
    const int cc = is_v ? c - CH : c;
    const uint4* from = static_cast<const uint4*>(is_v ? a.v_new : a.k_new) + src * CH + cc;
    uint4* to = static_cast<uint4*>(const_cast<void*>(is_v ? a.v_pool : a.k_pool)) + row * CH + cc;
    *to = __ldg(from);
  }
}

// Context length as the kernels use it: clamped to what the block table can
// address, with the clamp recorded in the status word.
__device__ __forceinline__ int checked_context(const DecodeArgs& a, int s, bool report) {
  int c = __ldg(a.context_lens + s);
  const int cap = min(a.max_blocks_per_seq * kBlock, a.max_context_len);
  if (c < 0 || c > cap) {
    if (report) flag_status(a.status, PA_DEV_BAD_CONTEXT);
    c = c < 0 ? 0 : cap;
  }
  return c;
}

}  // namespace pa
