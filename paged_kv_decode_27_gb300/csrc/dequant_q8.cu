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
// bf16 queries are converted to fp16 for the pass (exact for |q| in fp16's
// normal range: bf16 carries 8 significant bits) and its fp16 output back to
// bf16.
//
// One CTA per (sequence, block); a thread widens 16 codes of a row (one
// 16-byte load, two 16-byte stores) for K and then V.
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

__global__ void __launch_bounds__(256)
dequant_blocks_q8_kernel(const int8_t* __restrict__ k_codes, const int8_t* __restrict__ v_codes,
                         const float* __restrict__ k_scales, const float* __restrict__ v_scales,
                         const int32_t* __restrict__ block_tables, const int32_t* __restrict__ context_lens,
                         int max_blocks_per_seq, int num_kv_heads, int head_dim, int num_blocks, int B,
                         __half* __restrict__ k_out, __half* __restrict__ v_out, int32_t* __restrict__ table_out,
                         int* status) {
  grid_dependency_wait();   // the prompt's rows were appended by the kernel before us
  const int lb = blockIdx.x;
  const int s = blockIdx.y;
  const size_t ob = static_cast<size_t>(s) * B + lb;   // block of the copies
  if (threadIdx.x == 0) table_out[ob] = static_cast<int32_t>(ob);
  const int c = __ldg(context_lens + s);
  if (lb * kBlock >= c) return;
  const int id = __ldg(block_tables + static_cast<size_t>(s) * max_blocks_per_seq + lb);
  const bool live = id >= 0 && id < num_blocks;
  if (!live && threadIdx.x == 0) flag_status(status, PA_DEV_BAD_BLOCK_ID);
  const int chunks = head_dim / 16;                     // 16-code chunks per row
  const int per_block = num_kv_heads * kBlock * chunks; // chunks per (block, K or V)
  const size_t src0 = static_cast<size_t>(live ? id : 0) * num_kv_heads * kBlock;   // first row of the block
  const size_t dst0 = ob * num_kv_heads * kBlock;
  bool out_of_range = false;
  for (int i = threadIdx.x; i < 2 * per_block; i += blockDim.x) {
    const bool is_k = i < per_block;
    const int j = is_k ? i : i - per_block;
    const int row = j / chunks;                          // (head, slot) row within the block
    const int ch = j - row * chunks;
    uint4 lo = make_uint4(0u, 0u, 0u, 0u), hi = lo;
    // rows past the context (stale slots of the last block) are written as zeros
    if (live && lb * kBlock + row % kBlock < c) {
      const int8_t* codes = is_k ? k_codes : v_codes;
      const float* scales = is_k ? k_scales : v_scales;
      const uint4 w = __ldg(reinterpret_cast<const uint4*>(codes + (src0 + row) * head_dim) + ch);
      widen16(w, __ldg(scales + src0 + row), lo, hi, out_of_range);
    }
    uint4* dst = reinterpret_cast<uint4*>((is_k ? k_out : v_out) + (dst0 + row) * head_dim) + 2 * ch;
    dst[0] = lo;
    dst[1] = hi;
  }
  if (out_of_range) flag_status(status, PA_DEV_RANGE);
}

// Rows 0 .. cu_q_lens[num_seqs] - 1 of [rows][width] (width a multiple of 8)
// converted between bf16 and fp16: TO_HALF bf16 -> fp16 (clamped to fp16's
// range, reported), else fp16 -> bf16.
template <bool TO_HALF>
__global__ void __launch_bounds__(256)
convert_rows_kernel(const uint4* __restrict__ src, uint4* __restrict__ dst, const int32_t* __restrict__ cu_q_lens,
                    int num_seqs, int width, int* status) {
  grid_dependency_wait();
  const long long n = static_cast<long long>(__ldg(cu_q_lens + num_seqs)) * (width / 8);   // 8 values per uint4
  bool out_of_range = false;
  for (long long i = static_cast<long long>(blockIdx.x) * blockDim.x + threadIdx.x; i < n;
       i += static_cast<long long>(gridDim.x) * blockDim.x) {
    const uint4 v = src[i];
    const uint32_t w[4] = {v.x, v.y, v.z, v.w};
    uint32_t o[4];
#pragma unroll
    for (int k = 0; k < 4; ++k) {
      if constexpr (TO_HALF) {
        o[k] = pack_half_sat(__uint_as_float(w[k] << 16), __uint_as_float(w[k] & 0xffff0000u), out_of_range);
      } else {
        const __half2 h = *reinterpret_cast<const __half2*>(&w[k]);
        __nv_bfloat162 b = __floats2bfloat162_rn(__low2float(h), __high2float(h));
        o[k] = *reinterpret_cast<uint32_t*>(&b);
      }
    }
    dst[i] = make_uint4(o[0], o[1], o[2], o[3]);
  }
  if (out_of_range) flag_status(status, PA_DEV_RANGE);
}

}  // namespace

cudaError_t launch_dequant_q8(const void* k_codes, const void* v_codes, const float* k_scales,
                              const float* v_scales, const int32_t* block_tables, const int32_t* context_lens,
                              int num_seqs, int max_blocks_per_seq, int num_kv_heads, int head_dim,
                              int num_blocks, int B, void* k_out, void* v_out, int32_t* table_out, int* status,
                              cudaStream_t stream) {
  if (num_seqs == 0 || B == 0) return cudaSuccess;
  const dim3 grid(static_cast<unsigned>(B), static_cast<unsigned>(num_seqs));
  return launch_pdl(dequant_blocks_q8_kernel, grid, dim3(256), 0, stream, static_cast<const int8_t*>(k_codes),
                    static_cast<const int8_t*>(v_codes), k_scales, v_scales, block_tables, context_lens,
                    max_blocks_per_seq, num_kv_heads, head_dim, num_blocks, B, static_cast<__half*>(k_out),
                    static_cast<__half*>(v_out), table_out, status);
}

cudaError_t launch_convert_rows(const void* src, void* dst, const int32_t* cu_q_lens, int num_seqs, int width,
                                bool to_half, int* status, cudaStream_t stream) {
  int sms = device_sm_count();
  if (sms <= 0) sms = 152;
  const dim3 grid(static_cast<unsigned>(4 * sms));
  const uint4* s = static_cast<const uint4*>(src);
  uint4* d = static_cast<uint4*>(dst);
  return to_half ? launch_pdl(convert_rows_kernel<true>, grid, dim3(256), 0, stream, s, d, cu_q_lens, num_seqs, width,
                              status)
                 : launch_pdl(convert_rows_kernel<false>, grid, dim3(256), 0, stream, s, d, cu_q_lens, num_seqs, width,
                              status);
}

}  // namespace pa
