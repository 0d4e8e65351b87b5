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
// elements of each row; the eight rows' maxima come from one transposed
// butterfly that leaves row u's on lanes 4u .. 4u + 3, which compute its
// scale (so the division runs once for eight rows) and hand it to the other
// lanes; every lane writes its D/32 codes (so the 128- or 64-byte code row
// is one coalesced store) and lane 4u the float32 scale of row u.
//
// The scale is one IEEE division, s = amax / 127.  Each code is the
// round-to-nearest-even of the IEEE quotient fl(x / s), decided without a
// division in almost every case by a rounding test (Ziv's strategy: an
// approximation with a proven error bound fixes the result unless it lies
// within that bound of a decision boundary): t = x * (1/s) with the
// correctly rounded reciprocal is within 2^-16 of x / s for |x / s| <= 128,
// and fl(x / s) within 2^-17, so when t lies more than 2^-12 from a
// half-integer both round to the same integer; when some element of a row
// does not (or t is not finite), the warp recomputes that row's codes with
// the division itself.  Codes and scales are bit-exact functions of the row.
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

// Round-to-nearest-even of t = x * r (r = 1/s correctly rounded, s > 0):
// adding 1.5 * 2^23 leaves the nearest integer n of |t| < 2^22 in the low
// mantissa bits, so the low byte of the sum's bits is n in two's complement,
// and t - n (both exact) is the rounding error e in [-1/2, 1/2].  A finite t
// has |t| < 127.5 here (|x| <= amax, and r * amax = 127 within a few units in
// the last place; a subnormal s below 2^-128 makes r infinite), so "t not
// finite, or within the test's margin 2^-12 of a half-integer" is exactly
// !(|e| < 1/2 - 2^-12): a non-finite t gives a NaN e.  `near` is set then,
// when the division has to decide.  The explicit-rounding intrinsics keep
// the compiler from fusing the steps into FMAs.  Returns the sum's bits.
__device__ __forceinline__ uint32_t fast_code_bits(float x, float r, bool& near) {
  const float t = __fmul_rn(x, r);
  const float m = __fadd_rn(t, 12582912.f);
  const float e = __fsub_rn(t, __fsub_rn(m, 12582912.f));
  near |= !(fabsf(e) < 0.5f - 0x1p-12f);
  return __float_as_uint(m);
}

// the low bytes of EPL words as EPL packed codes
__device__ __forceinline__ uint32_t pack_codes(const uint32_t (&m)[4]) {
  return __byte_perm(__byte_perm(m[0], m[1], 0x0040u), __byte_perm(m[2], m[3], 0x0040u), 0x5410u);
}
__device__ __forceinline__ uint16_t pack_codes(const uint32_t (&m)[2]) {
  return static_cast<uint16_t>(__byte_perm(m[0], m[1], 0x0040u));
}

// the code itself: round-to-nearest-even of the IEEE quotient fl(x / s),
// clamped to [-127, 127]
__device__ __forceinline__ int exact_code(float x, float s) {
  const int c = __float2int_rn(__fdiv_rn(x, s));
  return c > 127 ? 127 : (c < -127 ? -127 : c);
}

template <typename T, int D>
__global__ void __launch_bounds__(256, 4)
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
    for (int u = 0; u < kHeadsPerPass; ++u) {
      raw[u] = In{};
      if (h0 + u < h_end) raw[u] = __ldcs(reinterpret_cast<const In*>(src + static_cast<size_t>(h0 + u) * D));
    }
    if (slot < 0) return;                                   // padding token
    if (slot >= static_cast<long long>(num_blocks) * kBlock) {
      if (lane == 0 && !is_v) flag_status(status, PA_DEV_BAD_SLOT);
      return;
    }
    const long long blk = slot / kBlock;
    const int off = static_cast<int>(slot - blk * kBlock);
    // this lane's elements and the partial maxima of its 8 rows (0 for rows
    // past the group)
    float x[kHeadsPerPass][EPL];
    float v[kHeadsPerPass];
#pragma unroll
    for (int u = 0; u < kHeadsPerPass; ++u) {
      const T* e = reinterpret_cast<const T*>(&raw[u]);
      v[u] = 0.f;
#pragma unroll
      for (int i = 0; i < EPL; ++i) {
        x[u][i] = h0 + u < h_end ? Elem<T>::to_f(e[i]) : 0.f;
        v[u] = fmaxf(v[u], fabsf(x[u][i]));
      }
    }
    // Row maxima by a transposed butterfly: at the exchanges over lane bits
    // 4, 3 and 2 each lane keeps half of its rows and receives the partner's
    // partial maxima of those rows, so that lane l ends with row
    // (l >> 2) & 7, whose maximum the exchanges over bits 1 and 0 complete
    // (9 shuffles for 8 rows).
    const bool b4 = (lane >> 4) & 1, b3 = (lane >> 3) & 1, b2 = (lane >> 2) & 1;
    float w4[4], w2[2];
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      const float keep = b4 ? v[4 + j] : v[j];
      const float send = b4 ? v[j] : v[4 + j];
      w4[j] = fmaxf(keep, __shfl_xor_sync(0xffffffffu, send, 16));
    }
#pragma unroll
    for (int j = 0; j < 2; ++j) {
      const float keep = b3 ? w4[2 + j] : w4[j];
      const float send = b3 ? w4[j] : w4[2 + j];
      w2[j] = fmaxf(keep, __shfl_xor_sync(0xffffffffu, send, 8));
    }
    float amax = fmaxf(b2 ? w2[1] : w2[0], __shfl_xor_sync(0xffffffffu, b2 ? w2[0] : w2[1], 4));
    amax = warp_max_xor(amax, 1, 2);
    // the scale of row (lane >> 2) & 7 and its reciprocal: one division for
    // the 8 rows
    const float sc_l = __fdiv_rn(amax, 127.f);
    const float rc_l = sc_l > 0.f ? __frcp_rn(sc_l) : 0.f;
    const int my_row = (lane >> 2) & 7;
    if ((lane & 3) == 0 && h0 + my_row < h_end)
      scales[(static_cast<size_t>(blk) * num_kv_heads + h0 + my_row) * kBlock + off] = sc_l;
#pragma unroll
    for (int u = 0; u < kHeadsPerPass; ++u) {
      const int h = h0 + u;
      if (h >= h_end) break;
      // r = 0 when s = 0 (an all-zero row, or amax / 127 below the subnormal
      // range): every finite element then gets code 0 on the fast path
      const float rc = __shfl_sync(0xffffffffu, rc_l, 4 * u);
      uint32_t m[EPL];
      bool near = false;
#pragma unroll
      for (int i = 0; i < EPL; ++i) m[i] = fast_code_bits(x[u][i], rc, near);
      if (__any_sync(0xffffffffu, near)) {   // rare: the row has a quotient near a tie
        const float sc = __shfl_sync(0xffffffffu, sc_l, 4 * u);
#pragma unroll
        for (int i = 0; i < EPL; ++i) m[i] = static_cast<uint32_t>(sc > 0.f ? exact_code(x[u][i], sc) : 0);
      }
      const size_t r = (static_cast<size_t>(blk) * num_kv_heads + h) * kBlock + off;
      reinterpret_cast<Out*>(codes + r * D)[lane] = pack_codes(m);
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
