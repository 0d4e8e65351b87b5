// prefill_umma.cu -- causal prompt attention over the paged pool on the 5th-
// generation tensor cores (tcgen05, accumulators in tensor memory).
//
// The prompt pass processes all prompt tokens at once (q_len = prompt length,
// "LLM Inference Server", Stage 1) under a causal mask ("LLM Inference Server
// From Scratch", What you build: fused attention with causal masking; How it
// works, 4 Attention Kernel: causal mask, GQA).  It is a dense contraction and
// compute-bound ("LLM Inference Server", What You Will Build), so it runs on
// tcgen05.mma:
//
//  * a 1-D grid over (128-row query tile, query head, sequence), the latest
//    (longest) query tiles first.  Six warps with fixed roles:
//      warps 0-3  softmax: thread r owns query row r of the tile.  It reads its
//                 row of S = Q K^T from tensor memory, applies the causal mask
//                 and the online softmax, writes its row of P (bf16/fp16) back
//                 into the same tensor-memory columns and, when its running
//                 max grows, rescales its row of O;
//      warp 4     TMA producer: K tiles and V tiles of 64 keys (4 pool blocks,
//                 read through the block table) into two separate 2-stage
//                 rings of 128-byte-swizzled shared memory;
//      warp 5     MMA issuer: S = Q K^T (M=128, N=64, K=D; Q and K from shared
//                 memory) and O += P V (M=128, N=D, K=64; P from tensor
//                 memory, V read MN-major straight from its pool layout).
//  * Tensor memory (256 columns per CTA, so two CTAs share an SM): two S/P
//    buffers of 64 columns and O (D columns).  S_{j+1} is computed while the
//    softmax works on S_j.
//  * A K stage is released as soon as its S MMA completes and a V stage when
//    its PV MMA completes, so K tiles stream ahead of the softmax; the
//    producer and the MMA issuer are event loops that act on whichever of
//    their inputs is ready first.
//  * O is rescaled lazily: only when a row's max grows by more than 2^8 (so
//    probabilities stay <= 256, exact in the final normalisation).
//  * Query i of a sequence with context c and q_len n sits at position
//    c - n + i and sees keys 0..c - n + i; value rows past the context are
//    zeroed in shared memory so stale pool data never reaches the output.
//
// Every wait is bounded; a timeout sets PA_DEV_WAIT_TIMEOUT, lets the copies
// and MMAs in flight finish (bounded) and frees the tensor memory.
#include <type_traits>

#include "pa_common.cuh"
#include "pa_internal.h"

namespace pa {

namespace {

constexpr int kRows = 128;     // query rows per CTA (MMA M)
constexpr int kKeys = 64;      // keys per K/V tile (4 pool blocks)
constexpr int kThreads = 192;  // 4 softmax warps + producer warp + MMA warp
constexpr int kTmemCols = 256;

template <int D>
struct UmmaLayout {
  static constexpr int NBOX = D / 64;                 // 128-byte column boxes per row
  static constexpr int Q_BYTES = kRows * D * 2;       // [NBOX][128 rows][128 B]
  static constexpr int KT_BYTES = kKeys * D * 2;      // one K (or V) tile: [NBOX][64 rows][128 B]
  static constexpr int K_OFF = Q_BYTES;               // K ring: 2 tiles
  static constexpr int V_OFF = Q_BYTES + 2 * KT_BYTES;  // V ring: 2 tiles
  static constexpr int SMEM = Q_BYTES + 4 * KT_BYTES;
  static constexpr int HALF_Q = kRows * 128;          // one 64-column box strip of Q
  static constexpr int HALF_KT = kKeys * 128;         // one 64-column box strip of K or V
  static constexpr uint32_t TMEM_S = 0;               // S/P buffers: 2 x kKeys columns
  static constexpr uint32_t TMEM_O = 2 * kKeys;       // O: D fp32 columns
};

}  // namespace

template <typename T, int D>
__global__ void __launch_bounds__(kThreads, 1)
prefill_umma_kernel(const __grid_constant__ CUtensorMap kmap, const __grid_constant__ CUtensorMap vmap,
                    const PrefillArgs a) {
  using L = UmmaLayout<D>;
  constexpr int NBOX = L::NBOX;
  constexpr bool kBf16 = !std::is_same<T, __half>::value;

  extern __shared__ uint8_t smem_raw[];
  // barriers: k_full[2] k_empty[2] v_full[2] v_empty[2] s_full[2] p_full[2] pv_done[2] o_done mma_final
  __shared__ __align__(8) uint64_t bars[16];
  __shared__ uint32_t tmem_base_sh;
  __shared__ volatile int abort_sh;
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                             ~static_cast<uintptr_t>(1023));
  const uint32_t sQ = smem_u32(smem);
  const uint32_t sK = sQ + L::K_OFF;
  const uint32_t sV = sQ + L::V_OFF;

  // heaviest query tiles first: tile index qt descends slowest over the 1-D grid
  const int per_layer = a.num_q_heads * a.num_seqs;
  const int qt = (gridDim.x / per_layer) - 1 - static_cast<int>(blockIdx.x) / per_layer;
  const int hq = static_cast<int>(blockIdx.x) % a.num_q_heads;
  const int s = (static_cast<int>(blockIdx.x) % per_layer) / a.num_q_heads;
  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const int G = a.num_q_heads / a.num_kv_heads;
  const int kvh = hq / G;

  grid_dependency_wait();   // the prompt's K/V were appended by the kernel before us
  const int q0 = __ldg(a.cu_q_lens + s);
  const int n = __ldg(a.cu_q_lens + s + 1) - q0;
  int c = __ldg(a.context_lens + s);
  const int cap = a.max_blocks_per_seq * kBlock;
  if (c < n || c > cap || n < 0 || n > a.max_q_len) {
    if (threadIdx.x == 0 && qt == 0 && hq == 0) flag_status(a.status, PA_DEV_BAD_CONTEXT);
    c = c > cap ? cap : c;
    if (c < n || n > a.max_q_len) return;
  }
  const int qrow0 = qt * kRows;
  if (qrow0 >= n) return;
  const int pos0 = c - n + qrow0;
  const int rows_cta = min(kRows, n - qrow0);
  const int n_kt = (pos0 + rows_cta - 1) / kKeys + 1;   // key tiles touching the causal range

  const uint32_t bar0 = smem_u32(&bars[0]);
  auto k_full = [&](int i) { return bar0 + 0u + 8u * i; };
  auto k_empty = [&](int i) { return bar0 + 16u + 8u * i; };
  auto v_full = [&](int i) { return bar0 + 32u + 8u * i; };
  auto v_empty = [&](int i) { return bar0 + 48u + 8u * i; };
  auto s_full = [&](int i) { return bar0 + 64u + 8u * i; };
  auto p_full = [&](int i) { return bar0 + 80u + 8u * i; };
  auto pv_done = [&](int i) { return bar0 + 96u + 8u * i; };
  const uint32_t o_done = bar0 + 112u, mma_final = bar0 + 120u;

  if (threadIdx.x == 0) {
    for (int i = 0; i < 2; ++i) {
      mbar_init(k_full(i), 1);
      mbar_init(k_empty(i), 1);
      mbar_init(v_full(i), 1);
      mbar_init(v_empty(i), 1);
      mbar_init(s_full(i), 1);
      mbar_init(p_full(i), 4);
      mbar_init(pv_done(i), 1);
    }
    mbar_init(o_done, 1);
    mbar_init(mma_final, 1);
    fence_barrier_init();
    abort_sh = 0;
  }
  if (warp == 0) {
    tmem_alloc(smem_u32(&tmem_base_sh), kTmemCols);
    tmem_relinquish();
  }
  // Q tile -> shared memory in the 128-byte-swizzled K-major layout
  if (warp < 4) {
    const int r = threadIdx.x;
    const int lr = qrow0 + r;
    const uint4* src = reinterpret_cast<const uint4*>(static_cast<const T*>(a.q) +
                                                      ((static_cast<size_t>(q0) + lr) * a.num_q_heads + hq) * D);
#pragma unroll
    for (int cc = 0; cc < D / 8; ++cc) {
      uint4 v = make_uint4(0u, 0u, 0u, 0u);
      if (lr < n) v = src[cc];
      const uint32_t dst = sQ + (cc >> 3) * L::HALF_Q + r * 128 + (((cc & 7) ^ (r & 7)) << 4);
      asm volatile("st.shared.v4.b32 [%0], {%1,%2,%3,%4};" ::"r"(dst), "r"(v.x), "r"(v.y), "r"(v.z), "r"(v.w)
                   : "memory");
    }
    fence_proxy_async_smem();
  }
  tc_fence_before_sync();
  __syncthreads();
  tc_fence_after_sync();
  const uint32_t tmem = tmem_base_sh;
  const uint32_t tO = tmem + L::TMEM_O;

  if (warp == 4) {
    // ------------------------------------------------------------ TMA producer
    if (lane == 0) {
      prefetch_tensormap(&kmap);
      prefetch_tensormap(&vmap);
      const uint64_t policy = l2_policy_evict_last();   // other heads of the group re-read these tiles
      const int oob_row = a.num_blocks * a.num_kv_heads * kBlock;   // rows past the pool read as zero
      auto tile_rows = [&](int j, int* y) {
#pragma unroll
        for (int b = 0; b < 4; ++b) {
          const int lb = j * 4 + b;
          y[b] = oob_row;
          if (lb * kBlock < c) {
            const int id = __ldg(a.block_tables + static_cast<size_t>(s) * a.max_blocks_per_seq + lb);
            if (id >= 0 && id < a.num_blocks)
              y[b] = (id * a.num_kv_heads + kvh) * kBlock;
            else
              flag_status(a.status, PA_DEV_BAD_BLOCK_ID);
          }
        }
      };
      auto load_tile = [&](const CUtensorMap* map, uint32_t dst, uint32_t bar, const int* y) {
        mbar_arrive_expect_tx(bar, L::KT_BYTES);
#pragma unroll
        for (int b = 0; b < 4; ++b)
#pragma unroll
          for (int h = 0; h < NBOX; ++h) tma_load_2d(dst + h * L::HALF_KT + b * 2048, map, h * 64, y[b], bar, policy);
      };
      int next_k = 0, next_v = 0;
      int yk[4], yv[4];
      tile_rows(0, yk);
      uint64_t t_last = global_timer_ns();
      for (uint32_t spin = 0; next_v < n_kt; ++spin) {
        bool progressed = false;
        if (next_k < n_kt && (next_k < 2 || mbar_test_wait(k_empty(next_k & 1), ((next_k - 2) >> 1) & 1))) {
          load_tile(&kmap, sK + (next_k & 1) * L::KT_BYTES, k_full(next_k & 1), yk);
          ++next_k;
          if (next_k < n_kt) tile_rows(next_k, yk);
          progressed = true;
        }
        if (next_v < next_k && (next_v < 2 || mbar_test_wait(v_empty(next_v & 1), ((next_v - 2) >> 1) & 1))) {
          tile_rows(next_v, yv);
          load_tile(&vmap, sV + (next_v & 1) * L::KT_BYTES, v_full(next_v & 1), yv);
          ++next_v;
          progressed = true;
        }
        if (progressed) {
          t_last = global_timer_ns();
        } else if ((spin & 63u) == 0 && (abort_sh || global_timer_ns() - t_last > 1000000000ull)) {
          abort_sh = 1;
          break;
        }
      }
      if (abort_sh) {
        // let the copies still in flight land before the CTA can exit
        for (int j = next_k - 2 < 0 ? 0 : next_k - 2; j < next_k; ++j)
          mbar_wait_bounded(k_full(j & 1), (j >> 1) & 1, 100000000ull);
        for (int j = next_v - 2 < 0 ? 0 : next_v - 2; j < next_v; ++j)
          mbar_wait_bounded(v_full(j & 1), (j >> 1) & 1, 100000000ull);
      }
    }
  } else if (warp == 5) {
    // --------------------------------------------------------------- MMA issuer
    const uint32_t id_s = umma_idesc_f16(kRows, kKeys, kBf16, false, false);
    const uint32_t id_o = umma_idesc_f16(kRows, D, kBf16, false, true);
    bool ok = true;
    int next_s = 0, next_pv = 0;
    uint64_t t_last = global_timer_ns();
    for (uint32_t spin = 0; next_pv < n_kt; ++spin) {
      bool progressed = false;
      // S_j = Q K_j^T into S buffer j%2 once K_j has landed and PV_{j-2} (which
      // read P_{j-2} from that buffer) has completed
      if (next_s < n_kt) {
        const int j = next_s;
        const bool ready = mbar_test_wait(k_full(j & 1), (j >> 1) & 1) &&
                           (j < 2 || mbar_test_wait(pv_done(j & 1), ((j - 2) >> 1) & 1));
        if (__all_sync(0xffffffffu, ready)) {
          tc_fence_after_sync();
          if (lane == 0) {
            const uint32_t kbase = sK + (j & 1) * L::KT_BYTES;
#pragma unroll
            for (int kk = 0; kk < D / 16; ++kk) {
              const uint64_t da = umma_desc_sw128(sQ + (kk >> 2) * L::HALF_Q + (kk & 3) * 32, 16, 1024);
              const uint64_t db = umma_desc_sw128(kbase + (kk >> 2) * L::HALF_KT + (kk & 3) * 32, 16, 1024);
              umma_f16(tmem + L::TMEM_S + (j & 1) * kKeys, da, db, id_s, kk > 0 ? 1u : 0u);
            }
            umma_commit(s_full(j & 1));
            umma_commit(k_empty(j & 1));
          }
          __syncwarp();
          ++next_s;
          progressed = true;
        }
      }
      // O += P_j V_j once the softmax has written P_j and V_j has landed
      if (next_pv < next_s) {
        const int j = next_pv;
        const bool ready = mbar_test_wait(p_full(j & 1), (j >> 1) & 1) &&
                           mbar_test_wait(v_full(j & 1), (j >> 1) & 1);
        if (__all_sync(0xffffffffu, ready)) {
          const uint32_t vbase = sV + (j & 1) * L::KT_BYTES;
          const int pb = c >> 4;
          if ((c & 15) && (pb >> 2) == j) {   // value rows past the context read as zero
            const int r0 = c & 15;
            for (int idx = lane; idx < (16 - r0) * NBOX * 8; idx += 32) {
              const int row = (pb & 3) * 16 + r0 + idx / (NBOX * 8);
              const int rem = idx % (NBOX * 8);
              const uint32_t addr = vbase + (rem >> 3) * L::HALF_KT + row * 128 + ((rem & 7) << 4);
              asm volatile("st.shared.v4.b32 [%0], {%1,%1,%1,%1};" ::"r"(addr), "r"(0u) : "memory");
            }
            fence_proxy_async_smem();
          }
          __syncwarp();
          tc_fence_after_sync();
          if (lane == 0) {
            const uint32_t pt = tmem + L::TMEM_S + (j & 1) * kKeys;   // P_j: 32 columns of packed pairs
#pragma unroll
            for (int kk = 0; kk < kKeys / 16; ++kk) {
              const uint64_t db = umma_desc_sw128(vbase + kk * 2048, L::HALF_KT, 1024);
              umma_f16_tmem_a(tO, pt + kk * 8, db, id_o, (j > 0 || kk > 0) ? 1u : 0u);
            }
            umma_commit(o_done);
            umma_commit(v_empty(j & 1));
            umma_commit(pv_done(j & 1));
          }
          __syncwarp();
          ++next_pv;
          progressed = true;
        }
      }
      if (progressed) {
        t_last = global_timer_ns();
      } else if ((spin & 63u) == 0) {
        const bool give_up = abort_sh || global_timer_ns() - t_last > 1000000000ull;
        if (__any_sync(0xffffffffu, give_up)) {
          ok = false;
          break;
        }
      }
    }
    if (!ok) abort_sh = 1;
    // every MMA issued by this warp has completed before the CTA tears down
    if (lane == 0) umma_commit(mma_final);
    mbar_wait_bounded(mma_final, 0, 100000000ull);
  } else {
    // ----------------------------------------------------------- softmax warps
    const int r = threadIdx.x;
    const int lr = qrow0 + r;
    const int pos = c - n + lr;                       // causal limit of this row
    const uint32_t lane_base = static_cast<uint32_t>(warp * 32) << 16;
    float m_used = -INFINITY;   // reference max of this row (log2 domain)
    float l = 0.f;              // sum of 2^(x - m_used)
    bool ok = true;
    // scale > 0 (the usual case): the max is taken on the raw scores and the
    // scale folds into one FMA per element; otherwise scale first.
    const bool pos_scale = a.scale_log2 > 0.f;
    const int warp_pos_min = c - n + qrow0 + warp * 32;   // smallest causal limit in this warp
    for (int j = 0; j < n_kt; ++j) {
      const uint32_t tbuf = tmem + L::TMEM_S + (j & 1) * kKeys + lane_base;
      ok = !abort_sh && mbar_wait_bounded(s_full(j & 1), (j >> 1) & 1);
      if (!__all_sync(0xffffffffu, ok)) {
        ok = false;
        break;
      }
      tc_fence_after_sync();
      float x[kKeys];
      tmem_ld64(tbuf, x);

      const int key0 = j * kKeys;
      if (!pos_scale) {
#pragma unroll
        for (int i = 0; i < kKeys; ++i) x[i] *= a.scale_log2;
      }
      if (key0 + kKeys - 1 > warp_pos_min) {   // a tile on the diagonal: causal mask
#pragma unroll
        for (int i = 0; i < kKeys; ++i)
          if (key0 + i > pos) x[i] = -INFINITY;
      }
      // row max as a tree (independent partial maxima)
      float pm[8];
#pragma unroll
      for (int k = 0; k < 8; ++k) pm[k] = fmaxf(x[k], x[k + 8]);
#pragma unroll
      for (int i = 16; i < kKeys; i += 8)
#pragma unroll
        for (int k = 0; k < 8; ++k) pm[k] = fmaxf(pm[k], x[i + k]);
      float mx = fmaxf(fmaxf(fmaxf(pm[0], pm[1]), fmaxf(pm[2], pm[3])),
                       fmaxf(fmaxf(pm[4], pm[5]), fmaxf(pm[6], pm[7])));
      if (pos_scale) mx *= a.scale_log2;
      const bool need = mx > m_used + 8.f;
      float factor = 1.f;
      if (need) {
        factor = exp2f(m_used - mx);   // 0 when m_used is still -inf
        l *= factor;
        m_used = mx;
      }
      if (j > 0 && __any_sync(0xffffffffu, need)) {
        // rescale this warp's rows of O once P_{j-1} V_{j-1} has landed
        ok = mbar_wait_bounded(o_done, (j - 1) & 1);
        if (!__all_sync(0xffffffffu, ok)) {
          ok = false;
          break;
        }
        tc_fence_after_sync();
#pragma unroll
        for (int cc = 0; cc < D / 32; ++cc) {
          float o[32];
          tmem_ld32(tO + lane_base + cc * 32, o);
#pragma unroll
          for (int i = 0; i < 32; ++i) o[i] *= factor;
          tmem_st32(tO + lane_base + cc * 32, o);
        }
      }
      const float mu = (m_used == -INFINITY) ? 0.f : m_used;
      const float sc = pos_scale ? a.scale_log2 : 1.f;   // p = 2^(x*sc - mu)
      float ps[8] = {0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f};   // independent partial sums
      uint32_t w[kKeys / 2];
#pragma unroll
      for (int i = 0; i < kKeys / 2; ++i) {
        const float p0 = fast_exp2(fmaf(x[2 * i], sc, -mu));
        const float p1 = fast_exp2(fmaf(x[2 * i + 1], sc, -mu));
        ps[(2 * i) & 7] += p0;
        ps[(2 * i + 1) & 7] += p1;
        w[i] = Mma<T>::pack(p0, p1);
      }
      l += ((ps[0] + ps[1]) + (ps[2] + ps[3])) + ((ps[4] + ps[5]) + (ps[6] + ps[7]));
      tmem_st32_u(tbuf, w);   // P_j over S_j: key 2i in the low half of column i
      tmem_wait_st();
      tc_fence_before_sync();
      __syncwarp();
      if (lane == 0) mbar_arrive(p_full(j & 1));
    }
    if (!ok) {
      abort_sh = 1;
    } else {
      ok = mbar_wait_bounded(o_done, (n_kt - 1) & 1);
      if (__all_sync(0xffffffffu, ok)) {
        tc_fence_after_sync();
        const float inv = l > 0.f ? 1.f / l : 0.f;
        T* orow = static_cast<T*>(a.out) + ((static_cast<size_t>(q0) + lr) * a.num_q_heads + hq) * D;
#pragma unroll
        for (int cc = 0; cc < D / 32; ++cc) {
          float o[32];
          tmem_ld32(tO + lane_base + cc * 32, o);
          if (lr < n) {
#pragma unroll
            for (int e = 0; e < 4; ++e) {
              uint4 v;
              v.x = Mma<T>::pack(o[8 * e + 0] * inv, o[8 * e + 1] * inv);
              v.y = Mma<T>::pack(o[8 * e + 2] * inv, o[8 * e + 3] * inv);
              v.z = Mma<T>::pack(o[8 * e + 4] * inv, o[8 * e + 5] * inv);
              v.w = Mma<T>::pack(o[8 * e + 6] * inv, o[8 * e + 7] * inv);
              reinterpret_cast<uint4*>(orow + cc * 32)[e] = v;
            }
          }
        }
      } else {
        abort_sh = 1;
      }
    }
  }

  // ------------------------------------------------------------------ teardown
  tc_fence_before_sync();
  __syncthreads();
  if (threadIdx.x == 0 && abort_sh) flag_status(a.status, PA_DEV_WAIT_TIMEOUT);
  if (warp == 0) {
    tc_fence_after_sync();
    tmem_dealloc(tmem, kTmemCols);
  }
}

namespace {
template <typename T, int D>
cudaError_t launch_umma_t(const PrefillArgs& a, const CUtensorMap& kmap, const CUtensorMap& vmap,
                          cudaStream_t stream) {
  const int smem = UmmaLayout<D>::SMEM + 1024;
  auto kern = prefill_umma_kernel<T, D>;
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
  if (e != cudaSuccess) return e;
  const long long ctas = static_cast<long long>((a.max_q_len + kRows - 1) / kRows) * a.num_q_heads * a.num_seqs;
  if (ctas > 0x7fffffffLL) return cudaErrorInvalidConfiguration;
  return launch_pdl(kern, dim3(static_cast<unsigned>(ctas)), dim3(kThreads), smem, stream, kmap, vmap, a);
}
}  // namespace

cudaError_t launch_prefill_umma(const PrefillArgs& a, int dtype, const CUtensorMap& kmap,
                                const CUtensorMap& vmap, cudaStream_t stream) {
  if (dtype == PA_BF16) {
    return a.head_dim == 128 ? launch_umma_t<__nv_bfloat16, 128>(a, kmap, vmap, stream)
                             : launch_umma_t<__nv_bfloat16, 64>(a, kmap, vmap, stream);
  }
  return a.head_dim == 128 ? launch_umma_t<__half, 128>(a, kmap, vmap, stream)
                           : launch_umma_t<__half, 64>(a, kmap, vmap, stream);
}

}  // namespace pa
