// append_q8.cu -- quantise each step's new K/V rows into the INT8 cache.
//
// The cached K and V are quantised dynamically to int8 per token head ("LLM
// Inference Server", Optional Bonus Extensions: INT8 KV-Cache Quantization)
// with the symmetric absmax rule of its Required Mathematical Concepts:
// s = max|x| / 127, x_q = round(x / s).  Rows arrive through the slot mapping
// of the float append (slot = block*16 + offset, negative = skip).
//
// One warp per token, K or V, and group of heads: the group's head rows are
// loaded together, before the slot mapping is consulted, so a warp waits on
// one load latency per group (up to eight heads; smaller groups when the
// batch is too small to fill the GPU otherwise).  Each lane holds D/32
// elements of a row, the row maximum is a warp reduction, and every lane
// writes its D/32 codes (so the 128- or 64-byte code row is one coalesced
// store) while lane 0 writes the float32 scale.
//
// The scale is one IEEE division, s = amax / 127.  Each code is the
// round-to-nearest-even of the IEEE quotient fl(x / s), decided without a
// division in almost every case by a rounding test (Ziv's strategy: an
// approximation with a proven error bound fixes the result unless it lies
// within that bound of a decision boundary): t = x * (1/s) with the
// correctly rounded reciprocal is within 2^-16 of x / s for |x / s| <= 128,
// and fl(x / s) within 2^-17, so when t lies more than 2^-12 from a
// half-integer both round to the same integer; otherwise (and for a
// non-finite t) the code takes the division itself.  Codes and scales are
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

constexpr int kHeadsPerPass = 8;

// round-to-nearest-even of fl(x / s) clamped to [-127, 127], for s > 0 and
// r = 1/s correctly rounded (see the rounding test above)
__device__ __forceinline__ int code_of(float x, float s, float r) {
  const float t = x * r;
  const float f = t - floorf(t);   // within 2^-25 of the fraction of t
  int c;
  if (fabsf(t) < 256.f && fabsf(f - 0.5f) > 0x1p-12f)
    c = __float2int_rn(t);
  else
    c = __float2int_rn(__fdiv_rn(x, s));
  return c > 127 ? 127 : (c < -127 ? -127 : c);
}

template <typename T, int D>
__global__ void __launch_bounds__(256)
append_q8_kernel(int8_t* __restrict__ k_codes, int8_t* __restrict__ v_codes, float* __restrict__ k_scales,
                 float* __restrict__ v_scales, const int64_t* __restrict__ slot_mapping,
                 const T* __restrict__ k_new, const T* __restrict__ v_new, int num_tokens, int num_kv_heads,
                 int heads_per_warp, int num_blocks, int* status) {
  allow_dependents();   // the decode that follows waits for our writes itself
  constexpr int EPL = D / 32;
  using In = typename Lanes<EPL>::In;
  using Out = typename Lanes<EPL>::Out;
  const int lane = threadIdx.x & 31;
  const long long t = static_cast<long long>(blockIdx.x) * 8 + (threadIdx.x >> 5);   // token
  if (t >= num_tokens) return;
  const bool is_v = (blockIdx.y & 1) != 0;
  const int h_begin = static_cast<int>(blockIdx.y >> 1) * heads_per_warp;
  const int h_end = min(h_begin + heads_per_warp, num_kv_heads);
  const T* src = (is_v ? v_new : k_new) + static_cast<size_t>(t) * num_kv_heads * D + lane * EPL;
  const long long slot = __ldg(slot_mapping + t);
  int8_t* codes = is_v ? v_codes : k_codes;
  float* scales = is_v ? v_scales : k_scales;
  for (int h0 = h_begin; h0 < h_end; h0 += kHeadsPerPass) {
    In raw[kHeadsPerPass];
#pragma unroll
    for (int u = 0; u < kHeadsPerPass; ++u)
      if (h0 + u < h_end) raw[u] = __ldcs(reinterpret_cast<const In*>(src + static_cast<size_t>(h0 + u) * D));
    if (slot < 0) return;                                   // padding token
    if (slot >= static_cast<long long>(num_blocks) * kBlock) {
      if (lane == 0 && !is_v) flag_status(status, PA_DEV_BAD_SLOT);
      return;
    }
    const long long blk = slot / kBlock;
    const int off = static_cast<int>(slot - blk * kBlock);
#pragma unroll
    for (int u = 0; u < kHeadsPerPass; ++u) {
      const int h = h0 + u;
      if (h >= h_end) break;
      const T* e = reinterpret_cast<const T*>(&raw[u]);
      float x[EPL];
      float amax = 0.f;
#pragma unroll
      for (int i = 0; i < EPL; ++i) {
        x[i] = Elem<T>::to_f(e[i]);
        amax = fmaxf(amax, fabsf(x[i]));
      }
      amax = warp_max_xor(amax, 1, 16);
      const float sc = __fdiv_rn(amax, 127.f);
      const float rc = sc > 0.f ? __frcp_rn(sc) : 0.f;
      Out packed = 0;
#pragma unroll
      for (int i = 0; i < EPL; ++i) {
        const int c = sc > 0.f ? code_of(x[i], sc, rc) : 0;
        packed |= static_cast<Out>(static_cast<Out>(c & 0xff) << (8 * i));
      }
      const size_t r = (static_cast<size_t>(blk) * num_kv_heads + h) * kBlock + off;
      reinterpret_cast<Out*>(codes + r * D)[lane] = packed;
      if (lane == 0) scales[r] = sc;
    }
  }
}

cudaError_t launch_append_q8(void* k_codes, void* v_codes, float* k_scales, float* v_scales,
                             const int64_t* slot_mapping, const void* k_new, const void* v_new, int num_tokens,
                             int num_kv_heads, int head_dim, int act_dtype, int num_blocks, int* status,
                             cudaStream_t stream) {
  if (num_tokens == 0) return cudaSuccess;
  const long long blocks = (static_cast<long long>(num_tokens) + 7) / 8;   // a warp per token and head group
  if (blocks > 0x7fffffffLL) return cudaErrorInvalidValue;
  // the largest head group (up to 8) that still gives ~16 warps per SM
  int sms = device_sm_count();
  if (sms <= 0) sms = 152;
  int hpw = 8;
  while (hpw > 1 && static_cast<long long>(num_tokens) * 2 * ((num_kv_heads + hpw - 1) / hpw) < 16LL * sms) hpw >>= 1;
  const int groups = (num_kv_heads + hpw - 1) / hpw;
  if (2LL * groups > 65535) return cudaErrorInvalidValue;
  dim3 grid(static_cast<unsigned>(blocks), static_cast<unsigned>(2 * groups));
  auto* kc = static_cast<int8_t*>(k_codes);
  auto* vc = static_cast<int8_t*>(v_codes);
  if (act_dtype == PA_BF16) {
    auto* kn = static_cast<const __nv_bfloat16*>(k_new);
    auto* vn = static_cast<const __nv_bfloat16*>(v_new);
    if (head_dim == 128)
      append_q8_kernel<__nv_bfloat16, 128><<<grid, 256, 0, stream>>>(kc, vc, k_scales, v_scales, slot_mapping, kn, vn,
                                                                      num_tokens, num_kv_heads, hpw, num_blocks, status);
    else
      append_q8_kernel<__nv_bfloat16, 64><<<grid, 256, 0, stream>>>(kc, vc, k_scales, v_scales, slot_mapping, kn, vn,
                                                                     num_tokens, num_kv_heads, hpw, num_blocks, status);
  } else {
    auto* kn = static_cast<const __half*>(k_new);
    auto* vn = static_cast<const __half*>(v_new);
    if (head_dim == 128)
      append_q8_kernel<__half, 128><<<grid, 256, 0, stream>>>(kc, vc, k_scales, v_scales, slot_mapping, kn, vn,
                                                               num_tokens, num_kv_heads, hpw, num_blocks, status);
    else
      append_q8_kernel<__half, 64><<<grid, 256, 0, stream>>>(kc, vc, k_scales, v_scales, slot_mapping, kn, vn,
                                                              num_tokens, num_kv_heads, hpw, num_blocks, status);
  }
  return cudaGetLastError();
}

}  // namespace pa
