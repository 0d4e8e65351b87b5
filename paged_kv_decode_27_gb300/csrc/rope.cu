// rope.cu -- rotary position embedding fused into the KV append.
//
// A fused attention path rotates K as it writes it ("Mini inference engine
// (KV cache + sampling + quantization)", Story / portfolio: fuse qkv_proj +
// RoPE + attention).  The rotation is the half-split form of the Llama family
// the pages build on: for position p, entries j and j + D/2 of a row turn by
// p * theta^(-2j/D).
//
//  * rope_cache_kernel: the (cos, sin) table [max_positions][D/2] of float2.
//    Angles and trigonometry run in float64 (a float32 angle p * f loses
//    ~1e-3 rad at p ~ 8K), the table stores float32.  Built once per model.
//  * append_kv_rope_kernel: the slot-mapped append of append_kv.cu, with each
//    K row rotated at its token's position on the way into the pool (fp32
//    arithmetic from the table, one rounding to the pool type); V is copied.
//    One thread per 16 bytes of the low half of a K row and the matching
//    16 bytes of the high half, so loads and stores stay 128-bit.
//  * apply_rope_kernel: the same rotation in place on rows [T][H][D] (the
//    queries of a step).
// A position outside [0, max_positions) skips its row and is reported in the
// status word (PA_DEV_BAD_POSITION).
#include "pa_common.cuh"
#include "pa_internal.h"

namespace pa {

namespace {

template <typename T> struct Vec;   // elements per 16-byte access
template <> struct Vec<float> { static constexpr int N = 4; };
template <> struct Vec<__nv_bfloat16> { static constexpr int N = 8; };
template <> struct Vec<__half> { static constexpr int N = 8; };

// Rotate the N pairs (lo[i], hi[i]) by the table entries cs[i] = (cos, sin).
template <typename T>
__device__ __forceinline__ void rotate16(uint4& lo, uint4& hi, const float2* cs) {
  constexpr int N = Vec<T>::N;
  T* l = reinterpret_cast<T*>(&lo);
  T* h = reinterpret_cast<T*>(&hi);
#pragma unroll
  for (int i = 0; i < N; ++i) {
    const float2 t = __ldg(cs + i);
    const float a = Elem<T>::to_f(l[i]);
    const float b = Elem<T>::to_f(h[i]);
    l[i] = Elem<T>::from_f(fmaf(a, t.x, -b * t.y));
    h[i] = Elem<T>::from_f(fmaf(b, t.x, a * t.y));
  }
}

}  // namespace

__global__ void __launch_bounds__(256)
rope_cache_kernel(float2* __restrict__ cache, int max_positions, int half, int head_dim, double theta) {
  const long long idx = static_cast<long long>(blockIdx.x) * blockDim.x + threadIdx.x;
  if (idx >= static_cast<long long>(max_positions) * half) return;
  const int p = static_cast<int>(idx / half);
  const int j = static_cast<int>(idx - static_cast<long long>(p) * half);
  const double inv = pow(theta, -2.0 * j / head_dim);
  double s, c;
  sincos(static_cast<double>(p) * inv, &s, &c);
  cache[idx] = make_float2(__double2float_rn(c), __double2float_rn(s));
}

template <typename T, int D>
__global__ void __launch_bounds__(256)
append_kv_rope_kernel(uint4* __restrict__ k_pool, uint4* __restrict__ v_pool, const int64_t* __restrict__ slot_mapping,
                      const int32_t* __restrict__ positions, const uint4* __restrict__ k_new,
                      const uint4* __restrict__ v_new, const float2* __restrict__ cache, int max_positions,
                      int num_tokens, int num_kv_heads, int num_blocks, int* status) {
  allow_dependents();   // the decode that follows waits for our writes itself
  constexpr int N = Vec<T>::N;
  constexpr int ROW = D * static_cast<int>(sizeof(T)) / 16;   // 16-byte chunks per row
  const bool is_v = blockIdx.y != 0;
  const int per_row = is_v ? ROW : ROW / 2;                   // K: one thread per (lo, hi) pair of chunks
  const long long idx = static_cast<long long>(blockIdx.x) * blockDim.x + threadIdx.x;
  if (idx >= static_cast<long long>(num_tokens) * num_kv_heads * per_row) return;
  const int c = static_cast<int>(idx % per_row);
  const long long th = idx / per_row;
  const int h = static_cast<int>(th % num_kv_heads);
  const long long t = th / num_kv_heads;

  const long long slot = __ldg(slot_mapping + t);
  if (slot < 0) return;
  if (slot >= static_cast<long long>(num_blocks) * kBlock) {
    if (c == 0 && h == 0 && !is_v) flag_status(status, PA_DEV_BAD_SLOT);
    return;
  }
  const long long blk = slot / kBlock;
  const int off = static_cast<int>(slot % kBlock);
  const size_t dst = ((static_cast<size_t>(blk) * num_kv_heads + h) * kBlock + off) * ROW;
  const size_t src = static_cast<size_t>(th) * ROW;
  if (is_v) {
    v_pool[dst + c] = __ldcs(v_new + src + c);
    return;
  }
  const int pos = __ldg(positions + t);
  if (pos < 0 || pos >= max_positions) {
    if (c == 0 && h == 0) flag_status(status, PA_DEV_BAD_POSITION);
    return;
  }
  uint4 lo = __ldcs(k_new + src + c);
  uint4 hi = __ldcs(k_new + src + ROW / 2 + c);
  rotate16<T>(lo, hi, cache + static_cast<size_t>(pos) * (D / 2) + c * N);
  k_pool[dst + c] = lo;
  k_pool[dst + ROW / 2 + c] = hi;
}

template <typename T, int D>
__global__ void __launch_bounds__(256)
apply_rope_kernel(uint4* __restrict__ x, const int32_t* __restrict__ positions, const float2* __restrict__ cache,
                  int max_positions, int num_tokens, int num_heads, int* status) {
  constexpr int N = Vec<T>::N;
  constexpr int ROW = D * static_cast<int>(sizeof(T)) / 16;
  constexpr int PER_ROW = ROW / 2;
  grid_dependency_wait();
  const long long idx = static_cast<long long>(blockIdx.x) * blockDim.x + threadIdx.x;
  if (idx >= static_cast<long long>(num_tokens) * num_heads * PER_ROW) return;
  const int c = static_cast<int>(idx % PER_ROW);
  const long long th = idx / PER_ROW;
  const long long t = th / num_heads;
  const int pos = __ldg(positions + t);
  if (pos < 0 || pos >= max_positions) {
    if (c == 0 && th == t * num_heads) flag_status(status, PA_DEV_BAD_POSITION);
    return;
  }
  const size_t row = static_cast<size_t>(th) * ROW;
  uint4 lo = x[row + c];
  uint4 hi = x[row + PER_ROW + c];
  rotate16<T>(lo, hi, cache + static_cast<size_t>(pos) * (D / 2) + c * N);
  x[row + c] = lo;
  x[row + PER_ROW + c] = hi;
}

// One switch over (dtype, head_dim) per kernel template.
#define PA_ROPE_DISPATCH(KERNEL, GRID, STREAM, ...)                                          \
  do {                                                                                        \
    if (dtype == PA_BF16) {                                                                   \
      if (head_dim == 128) KERNEL<__nv_bfloat16, 128><<<GRID, 256, 0, STREAM>>>(__VA_ARGS__); \
      else KERNEL<__nv_bfloat16, 64><<<GRID, 256, 0, STREAM>>>(__VA_ARGS__);                  \
    } else if (dtype == PA_F16) {                                                             \
      if (head_dim == 128) KERNEL<__half, 128><<<GRID, 256, 0, STREAM>>>(__VA_ARGS__);        \
      else KERNEL<__half, 64><<<GRID, 256, 0, STREAM>>>(__VA_ARGS__);                         \
    } else {                                                                                  \
      if (head_dim == 128) KERNEL<float, 128><<<GRID, 256, 0, STREAM>>>(__VA_ARGS__);         \
      else KERNEL<float, 64><<<GRID, 256, 0, STREAM>>>(__VA_ARGS__);                          \
    }                                                                                         \
  } while (0)

cudaError_t launch_rope_cache(float* cos_sin, int max_positions, int head_dim, double theta, cudaStream_t stream) {
  const int half = head_dim / 2;
  const long long n = static_cast<long long>(max_positions) * half;
  if (n == 0) return cudaSuccess;
  const long long blocks = (n + 255) / 256;
  if (blocks > 0x7fffffffLL) return cudaErrorInvalidValue;
  rope_cache_kernel<<<static_cast<unsigned>(blocks), 256, 0, stream>>>(reinterpret_cast<float2*>(cos_sin),
                                                                      max_positions, half, head_dim, theta);
  return cudaGetLastError();
}

cudaError_t launch_append_rope(void* k_pool, void* v_pool, const int64_t* slot_mapping, const int32_t* positions,
                               const void* k_new, const void* v_new, const float* cos_sin, int max_positions,
                               int num_tokens, int num_kv_heads, int head_dim, int dtype, int num_blocks,
                               int* status, cudaStream_t stream) {
  if (num_tokens == 0) return cudaSuccess;
  const int row = head_dim * (dtype == PA_F32 ? 4 : 2) / 16;
  const long long per_tensor = static_cast<long long>(num_tokens) * num_kv_heads * row;   // V threads (K: half)
  const long long blocks = (per_tensor + 255) / 256;
  if (blocks > 0x7fffffffLL) return cudaErrorInvalidValue;
  dim3 grid(static_cast<unsigned>(blocks), 2);
  PA_ROPE_DISPATCH(append_kv_rope_kernel, grid, stream, static_cast<uint4*>(k_pool), static_cast<uint4*>(v_pool),
                   slot_mapping, positions, static_cast<const uint4*>(k_new), static_cast<const uint4*>(v_new),
                   reinterpret_cast<const float2*>(cos_sin), max_positions, num_tokens, num_kv_heads, num_blocks,
                   status);
  return cudaGetLastError();
}

cudaError_t launch_apply_rope(void* x, const int32_t* positions, const float* cos_sin, int max_positions,
                              int num_tokens, int num_heads, int head_dim, int dtype, int* status,
                              cudaStream_t stream) {
  if (num_tokens == 0) return cudaSuccess;
  const int per_row = head_dim * (dtype == PA_F32 ? 4 : 2) / 32;
  const long long n = static_cast<long long>(num_tokens) * num_heads * per_row;
  const long long blocks = (n + 255) / 256;
  if (blocks > 0x7fffffffLL) return cudaErrorInvalidValue;
  const dim3 grid(static_cast<unsigned>(blocks));
  PA_ROPE_DISPATCH(apply_rope_kernel, grid, stream, static_cast<uint4*>(x), positions,
                   reinterpret_cast<const float2*>(cos_sin), max_positions, num_tokens, num_heads, status);
  return cudaGetLastError();
}

}  // namespace pa
