// append_q8.cu -- quantise each step's new K/V rows into the INT8 cache.
//
// The cached K and V are quantised dynamically to int8 per token head ("LLM
// Inference Server", Optional Bonus Extensions: INT8 KV-Cache Quantization)
// with the symmetric absmax rule of its Required Mathematical Concepts:
// s = max|x| / 127, x_q = round(x / s).  Rows arrive through the slot mapping
// of the float append (slot = block*16 + offset, negative = skip).
//
// One warp per (token, head) row of K or V: each lane holds D/32 elements,
// the row maximum is a warp reduction, and every lane writes its D/32 codes
// (so the 128- or 64-byte code row is one coalesced store) while lane 0
// writes the float32 scale.  The scale and each x / s are single IEEE
// divisions and the rounding is to nearest even, so codes and scales are
// bit-exact functions of the row.
#include "pa_common.cuh"
#include "pa_internal.h"

namespace pa {

namespace {

template <int N> struct Lanes;
template <> struct Lanes<4> {   // D = 128: 8 bytes in, 4 codes out per lane
  using In = uint2;
  using Out = uint32_t;
};
template <> struct Lanes<2> {   // D = 64: 4 bytes in, 2 codes out per lane
  using In = uint32_t;
  using Out = uint16_t;
};

}  // namespace

template <typename T, int D>
__global__ void __launch_bounds__(256)
append_q8_kernel(int8_t* __restrict__ k_codes, int8_t* __restrict__ v_codes, float* __restrict__ k_scales,
                 float* __restrict__ v_scales, const int64_t* __restrict__ slot_mapping,
                 const T* __restrict__ k_new, const T* __restrict__ v_new, int num_tokens, int num_kv_heads,
                 int num_blocks, int* status) {
  allow_dependents();   // the decode that follows waits for our writes itself
  constexpr int EPL = D / 32;
  using In = typename Lanes<EPL>::In;
  using Out = typename Lanes<EPL>::Out;
  const int lane = threadIdx.x & 31;
  const long long row = static_cast<long long>(blockIdx.x) * 8 + (threadIdx.x >> 5);
  if (row >= static_cast<long long>(num_tokens) * num_kv_heads) return;
  const bool is_v = blockIdx.y != 0;
  const long long t = row / num_kv_heads;
  const int h = static_cast<int>(row - t * num_kv_heads);

  const long long slot = __ldg(slot_mapping + t);
  if (slot < 0) return;                                   // padding token
  if (slot >= static_cast<long long>(num_blocks) * kBlock) {
    if (lane == 0 && h == 0 && !is_v) flag_status(status, PA_DEV_BAD_SLOT);
    return;
  }

  const T* src = (is_v ? v_new : k_new) + static_cast<size_t>(row) * D + lane * EPL;
  const In raw = __ldcs(reinterpret_cast<const In*>(src));
  const T* e = reinterpret_cast<const T*>(&raw);
  float x[EPL];
  float amax = 0.f;
#pragma unroll
  for (int i = 0; i < EPL; ++i) {
    x[i] = Elem<T>::to_f(e[i]);
    amax = fmaxf(amax, fabsf(x[i]));
  }
  amax = warp_max_xor(amax, 1, 16);
  const float s = __fdiv_rn(amax, 127.f);

  Out packed = 0;
#pragma unroll
  for (int i = 0; i < EPL; ++i) {
    int c = 0;
    if (s > 0.f) {
      c = __float2int_rn(__fdiv_rn(x[i], s));
      c = c > 127 ? 127 : (c < -127 ? -127 : c);
    }
    packed |= static_cast<Out>(static_cast<Out>(c & 0xff) << (8 * i));
  }
  const long long blk = slot / kBlock;
  const int off = static_cast<int>(slot - blk * kBlock);
  const size_t r = (static_cast<size_t>(blk) * num_kv_heads + h) * kBlock + off;
  int8_t* codes = is_v ? v_codes : k_codes;
  reinterpret_cast<Out*>(codes + r * D)[lane] = packed;
  if (lane == 0) (is_v ? v_scales : k_scales)[r] = s;
}

cudaError_t launch_append_q8(void* k_codes, void* v_codes, float* k_scales, float* v_scales,
                             const int64_t* slot_mapping, const void* k_new, const void* v_new, int num_tokens,
                             int num_kv_heads, int head_dim, int act_dtype, int num_blocks, int* status,
                             cudaStream_t stream) {
  if (num_tokens == 0) return cudaSuccess;
  const long long rows = static_cast<long long>(num_tokens) * num_kv_heads;
  const long long blocks = (rows + 7) / 8;
  if (blocks > 0x7fffffffLL) return cudaErrorInvalidValue;
  dim3 grid(static_cast<unsigned>(blocks), 2);
  auto* kc = static_cast<int8_t*>(k_codes);
  auto* vc = static_cast<int8_t*>(v_codes);
  if (act_dtype == PA_BF16) {
    auto* kn = static_cast<const __nv_bfloat16*>(k_new);
    auto* vn = static_cast<const __nv_bfloat16*>(v_new);
    if (head_dim == 128)
      append_q8_kernel<__nv_bfloat16, 128><<<grid, 256, 0, stream>>>(kc, vc, k_scales, v_scales, slot_mapping, kn, vn,
                                                                      num_tokens, num_kv_heads, num_blocks, status);
    else
      append_q8_kernel<__nv_bfloat16, 64><<<grid, 256, 0, stream>>>(kc, vc, k_scales, v_scales, slot_mapping, kn, vn,
                                                                     num_tokens, num_kv_heads, num_blocks, status);
  } else {
    auto* kn = static_cast<const __half*>(k_new);
    auto* vn = static_cast<const __half*>(v_new);
    if (head_dim == 128)
      append_q8_kernel<__half, 128><<<grid, 256, 0, stream>>>(kc, vc, k_scales, v_scales, slot_mapping, kn, vn,
                                                               num_tokens, num_kv_heads, num_blocks, status);
    else
      append_q8_kernel<__half, 64><<<grid, 256, 0, stream>>>(kc, vc, k_scales, v_scales, slot_mapping, kn, vn,
                                                              num_tokens, num_kv_heads, num_blocks, status);
  }
  return cudaGetLastError();
}

}  // namespace pa
