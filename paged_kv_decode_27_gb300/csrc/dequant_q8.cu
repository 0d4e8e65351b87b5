// dequant_q8.cu -- the blocks of a prompt pass over an INT8 cache, dequantised
// into a float pool for the tcgen05 prompt pass.
//
// The prompt pass processes all prompt tokens at once ("LLM Inference Server",
// Stage 1) and is compute-bound, so over an INT8 cache ("LLM Inference Server",
// Optional Bonus Extensions: INT8 KV-Cache Quantization: x_hat = s * x_q) it
// reads each sequence's blocks once here and runs the fp16 prompt pass over
// the copies: the copies cost ~3x the codes' bytes of traffic against the
// pass's dense products.
//
// Layout of the copies: a pool of num_seqs * B blocks in the float pool layout
// [block][H_kv][16][D] (fp16), sequence s owning blocks s * B .. s * B + B - 1
// in order (B = blocks of the longest context), and its block table
// table[s][lb] = s * B + lb.  Row (s, lb, h, r) holds s_row * code rounded once
// to fp16 (11 significant bits), where s_row and the codes are those of block
// block_tables[s][lb]; a value past fp16's range is clamped to +-65504 and
// reported (PA_DEV_RANGE).  Rows past a sequence's context are zeros, and
// blocks past it are not written (the prompt pass never reads them); a block id
// outside the pool is reported and its copy holds zeros.
//
// bf16 queries are converted to fp16 by the pass itself (in shared memory,
// exact for |q| in fp16's normal range: bf16 carries 8 significant bits),
// which also stores its output rows as bf16.
//
// One CTA per (sequence, block); a thread widens 16 codes of a row (one
// 16-byte load, two 16-byte stores), eight such chunks with their loads
// issued together, and the context length and block id are read together:
// a CTA waits on two load latencies.
#include "pa_common.cuh"
#include "pa_internal.h"

namespace pa {

namespace {

constexpr float kHalfMax = 65504.f;

// two floats as fp16, clamped to fp16's range; `out` records a clamp
__device__ __forceinline__ uint32_t pack_half_sat(float a, float b, bool& out) {
  out |= !(fabsf(a) <= kHalfMax) || !(fabsf(b) <= kHalfMax);
  __half2 v = __floats2half2_rn(fminf(fmaxf(a, -kHalfMax), kHalfMax), fminf(fmaxf(b, -kHalfMax), kHalfMax));
  return *reinterpret_cast<uint32_t*>(&v);
}

// 16 codes (4 words) times the row scale, as 16 fp16 values (8 words)
__device__ __forceinline__ void widen16(const uint4 w, float s, uint4& lo, uint4& hi, bool& out) {
  const uint32_t wv[4] = {w.x, w.y, w.z, w.w};
  uint32_t o[8];
#pragma unroll
  for (int k = 0; k < 4; ++k) {
    const int32_t x = static_cast<int32_t>(wv[k]);
    // bytes 0..3 of the word as signed integers (arithmetic shifts extend the sign)
    const float c0 = static_cast<float>((x << 24) >> 24);
    const float c1 = static_cast<float>((x << 16) >> 24);
    const float c2 = static_cast<float>((x << 8) >> 24);
    const float c3 = static_cast<float>(x >> 24);
    o[2 * k] = pack_half_sat(s * c0, s * c1, out);
    o[2 * k + 1] = pack_half_sat(s * c2, s * c3, out);
  }
  lo = make_uint4(o[0], o[1], o[2], o[3]);
  hi = make_uint4(o[4], o[5], o[6], o[7]);
}

constexpr int kUnrollBlock = 8;   // chunks a thread loads before widening the first

__device__ __forceinline__ void dequant_block(const DequantQ8Args& a, int s, int lb) {
  const size_t ob = static_cast<size_t>(s) * a.B + lb;   // block of the copies
  const int c = __ldg(a.context_lens + s);
  // lb < B <= max_blocks_per_seq: inside the sequence's table row
  const int id = __ldg(a.block_tables + static_cast<size_t>(s) * a.max_blocks_per_seq + lb);
  if (threadIdx.x == 0) a.table_out[ob] = static_cast<int32_t>(ob);
  if (lb * kBlock >= c) return;
  const bool live = id >= 0 && id < a.num_blocks;
  if (!live && threadIdx.x == 0) flag_status(a.status, PA_DEV_BAD_BLOCK_ID);
  const int chunks = a.head_dim / 16;                     // 16-code chunks per row
  const int per_block = a.num_kv_heads * kBlock * chunks; // chunks per (block, K or V)
  const size_t src0 = static_cast<size_t>(live ? id : 0) * a.num_kv_heads * kBlock;   // first row of the block
  const size_t dst0 = ob * a.num_kv_heads * kBlock;
  const int valid = c - lb * kBlock;                      // rows of the block inside the context
  const bool out32 = ((reinterpret_cast<uintptr_t>(a.k_out) | reinterpret_cast<uintptr_t>(a.v_out)) & 31u) == 0;
  bool out_of_range = false;
  for (int base = 0; base < 2 * per_block; base += kUnrollBlock * blockDim.x) {
    uint4 w[kUnrollBlock];
    float sc[kUnrollBlock];
#pragma unroll
    for (int u = 0; u < kUnrollBlock; ++u) {
      const int i = base + u * blockDim.x + threadIdx.x;
      const bool is_k = i < per_block;
      const int j = is_k ? i : i - per_block;
      const int row = j / chunks;                        // (head, slot) row within the block
      // rows past the context (stale slots of the last block) are written as zeros
      if (i < 2 * per_block && live && row % kBlock < valid) {
        const int8_t* codes = is_k ? a.k_codes : a.v_codes;
        const float* scales = is_k ? a.k_scales : a.v_scales;
        w[u] = __ldg(reinterpret_cast<const uint4*>(codes + (src0 + row) * a.head_dim) + (j - row * chunks));
        sc[u] = __ldg(scales + src0 + row);
      } else {
        w[u] = make_uint4(0u, 0u, 0u, 0u);
        sc[u] = 0.f;
      }
    }
#pragma unroll
    for (int u = 0; u < kUnrollBlock; ++u) {
      const int i = base + u * blockDim.x + threadIdx.x;
      if (i >= 2 * per_block) break;
      const bool is_k = i < per_block;
      const int j = is_k ? i : i - per_block;
      const int row = j / chunks;
      uint4 lo, hi;
      widen16(w[u], sc[u], lo, hi, out_of_range);
      uint4* dst = reinterpret_cast<uint4*>(static_cast<__half*>(is_k ? a.k_out : a.v_out) + (dst0 + row) * a.head_dim) +
                   2 * (j - row * chunks);
      if (out32) {
        // one whole 32-byte sector (the copies are 32-byte aligned when their base is)
        asm volatile("st.global.v8.b32 [%0], {%1,%2,%3,%4,%5,%6,%7,%8};" ::"l"(dst), "r"(lo.x), "r"(lo.y), "r"(lo.z),
                     "r"(lo.w), "r"(hi.x), "r"(hi.y), "r"(hi.z), "r"(hi.w)
                     : "memory");
      } else {
        dst[0] = lo;
        dst[1] = hi;
      }
    }
  }
  if (out_of_range) flag_status(a.status, PA_DEV_RANGE);
}

__global__ void __launch_bounds__(256) dequant_blocks_q8_kernel(const DequantQ8Args a) {
  grid_dependency_wait();   // the prompt's rows were appended by the kernel before us
  dequant_block(a, static_cast<int>(blockIdx.y), static_cast<int>(blockIdx.x));
}

}  // namespace

cudaError_t launch_dequant_q8(const DequantQ8Args& a, cudaStream_t stream) {
  if (a.num_seqs == 0 || a.B == 0) return cudaSuccess;
  return launch_pdl(dequant_blocks_q8_kernel, dim3(static_cast<unsigned>(a.B), static_cast<unsigned>(a.num_seqs)),
                    dim3(256), 0, stream, a);
}

}  // namespace pa
