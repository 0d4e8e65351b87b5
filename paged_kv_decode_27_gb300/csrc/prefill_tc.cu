// prefill_tc.cu -- causal prompt attention over the paged pool (bf16 / fp16).
//
// The prompt pass of an inference engine processes all prompt tokens at once
// (q_len = prompt length, "LLM Inference Server", Stage 1) with a causal mask
// ("LLM Inference Server From Scratch", What you build: fused attention with
// causal masking; How it works, 4 Attention Kernel: causal mask, GQA).  It is
// compute-bound, so it runs as tensor-core tiles:
//
//  * grid = (query tile of 64 rows, query head, sequence); the longest query
//    tiles (latest positions, most keys) are scheduled first.
//  * 4 warps x 16 query rows.  Key/value tiles of 64 positions (4 pool blocks)
//    are fetched by TMA from the block table into an NS-stage ring of
//    128-byte-swizzled shared memory; one thread issues, one mbarrier per
//    stage, a CTA barrier before a stage is refilled.
//  * S = Q K^T and O += P V with mma.sync m16n8k16 (fp32 accumulate), fp32
//    online softmax in the log2 domain, P reused from the S accumulators as the
//    A operand, V read through ldmatrix.trans.
//  * Query i of sequence s sits at position c - q_len + i; key k is visible iff
//    k <= that position.  Value rows past the context are zeroed so stale pool
//    data never reaches the output.
#include "pa_common.cuh"
#include "pa_internal.h"

namespace pa {

template <typename T, int D, int NS>
__global__ void __launch_bounds__(128)
prefill_tc_kernel(const __grid_constant__ CUtensorMap kmap, const __grid_constant__ CUtensorMap vmap,
                  const PrefillArgs a) {
  constexpr int BQ = 64;               // query rows per CTA
  constexpr int BK = 64;               // key positions per tile (4 pool blocks)
  constexpr int NBOX = D / 64;
  constexpr int BOX = 16 * 128;
  constexpr int BLKT = NBOX * BOX;     // one pool block of K (or V) for one head
  constexpr int KT = 4 * BLKT;         // 64 keys of K (or V)
  constexpr int STAGE = 2 * KT;
  constexpr int KS = D / 16;           // k-steps of Q K^T
  constexpr int NTS = BK / 8;          // n-tiles of S
  constexpr int NTO = D / 8;           // n-tiles of O

  extern __shared__ uint8_t smem_raw[];
  __shared__ __align__(8) uint64_t bars[NS];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                             ~static_cast<uintptr_t>(1023));

  const int qt = gridDim.x - 1 - blockIdx.x;
  const int hq = blockIdx.y;
  const int s = blockIdx.z;
  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const int g = lane >> 2;
  const int tq = lane & 3;
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
    if (c < n) return;   // nothing sensible to compute for this sequence
  }
  const int qrow0 = qt * BQ;
  if (qrow0 >= n) return;
  const int pos0 = c - n + qrow0;                        // position of the CTA's first row
  const int rows_cta = min(BQ, n - qrow0);
  const int n_kt = (pos0 + rows_cta - 1) / BK + 1;       // key tiles touching the causal range

  const uint32_t sbase = smem_u32(smem);
  const uint32_t bar0 = smem_u32(&bars[0]);
  const uint64_t policy = l2_policy_evict_last();        // K/V tiles are re-read by other heads
  if (threadIdx.x == 0) {
    for (int st = 0; st < NS; ++st) mbar_init(bar0 + 8 * st, 1);
    fence_barrier_init();
  }
  __syncthreads();

  const int oob_row = a.num_blocks * a.num_kv_heads * kBlock;   // TMA zero-fills rows >= this
  auto issue = [&](int kt) {   // thread 0 only
    const int st = kt % NS;
    const uint32_t bar = bar0 + 8 * st;
    const uint32_t dst = sbase + st * STAGE;
    mbar_arrive_expect_tx(bar, STAGE);
#pragma unroll
    for (int b = 0; b < 4; ++b) {
      const int lb = kt * 4 + b;
      int y = oob_row;
      if (lb * kBlock < c) {
        const int id = __ldg(a.block_tables + static_cast<size_t>(s) * a.max_blocks_per_seq + lb);
        if (id >= 0 && id < a.num_blocks) {
          y = (id * a.num_kv_heads + kvh) * kBlock;
        } else {
          flag_status(a.status, PA_DEV_BAD_BLOCK_ID);
        }
      }
#pragma unroll
      for (int nb = 0; nb < NBOX; ++nb) {
        tma_load_2d(dst + b * BLKT + nb * BOX, &kmap, nb * 64, y, bar, policy);
        tma_load_2d(dst + KT + b * BLKT + nb * BOX, &vmap, nb * 64, y, bar, policy);
      }
    }
  };
  if (threadIdx.x == 0) {
    prefetch_tensormap(&kmap);
    prefetch_tensormap(&vmap);
    for (int kt = 0; kt < NS && kt < n_kt; ++kt) issue(kt);
  }

  // Q fragments (A operand: rows = this warp's 16 queries, k = head dim)
  const int lr0 = qrow0 + warp * 16 + g;      // local query index of fragment row g
  const int lr1 = lr0 + 8;
  uint32_t qa[KS][4];
  {
    const T* qb = static_cast<const T*>(a.q);
    const size_t r0 = (static_cast<size_t>(q0) + lr0) * a.num_q_heads + hq;
    const size_t r1 = (static_cast<size_t>(q0) + lr1) * a.num_q_heads + hq;
#pragma unroll
    for (int ks = 0; ks < KS; ++ks) {
      const int d = ks * 16 + 2 * tq;
      qa[ks][0] = lr0 < n ? *reinterpret_cast<const uint32_t*>(qb + r0 * D + d) : 0u;
      qa[ks][1] = lr1 < n ? *reinterpret_cast<const uint32_t*>(qb + r1 * D + d) : 0u;
      qa[ks][2] = lr0 < n ? *reinterpret_cast<const uint32_t*>(qb + r0 * D + d + 8) : 0u;
      qa[ks][3] = lr1 < n ? *reinterpret_cast<const uint32_t*>(qb + r1 * D + d + 8) : 0u;
    }
  }
  const int pos_r0 = c - n + lr0;             // causal limits of the two fragment rows
  const int pos_r1 = pos_r0 + 8;
  const int warp_pos_max = c - n + min(qrow0 + warp * 16 + 15, n - 1);
  const bool warp_active = qrow0 + warp * 16 < n;   // warp-uniform: mma/ldmatrix are .sync

  float m_run[2] = {-INFINITY, -INFINITY};
  float l_run[2] = {0.f, 0.f};
  float o[NTO][4];
#pragma unroll
  for (int j = 0; j < NTO; ++j) o[j][0] = o[j][1] = o[j][2] = o[j][3] = 0.f;

  const int kb_row = (lane & 7) + (lane >> 4) * 8;        // K rows for ldmatrix (B of S)
  const int kb_chk = (lane >> 3) & 1;
  const int vb_row = (lane & 7) + ((lane >> 3) & 1) * 8;  // V rows for ldmatrix.trans (B of O)
  const int vb_chk = lane >> 4;

  int fail_kt = -1;
  for (int kt = 0; kt < n_kt; ++kt) {
    const int st = kt % NS;
    const bool got = mbar_wait_bounded(bar0 + 8 * st, (kt / NS) & 1);
    if (!__syncthreads_and(got)) {
      fail_kt = kt;
      break;
    }
    const int key0 = kt * BK;
    if (warp_active && key0 <= warp_pos_max) {
      const uint32_t kt_s = sbase + st * STAGE;
      const uint32_t vt_s = kt_s + KT;
      // ---- S = Q K^T ------------------------------------------------------
      float sc[NTS][4];
#pragma unroll
      for (int j = 0; j < NTS; ++j) sc[j][0] = sc[j][1] = sc[j][2] = sc[j][3] = 0.f;
#pragma unroll
      for (int ks = 0; ks < KS; ++ks) {
        const int ch = 2 * ks + kb_chk;
#pragma unroll
        for (int np = 0; np < NTS / 2; ++np) {
          const int kr = np * 16 + kb_row;
          uint32_t b0, b1, b2, b3;
          ldsm_x4(kt_s + (kr >> 4) * BLKT + (ch >> 3) * BOX + swz128(kr & 15, ch & 7), b0, b1, b2, b3);
          Mma<T>::run(sc[2 * np], qa[ks], b0, b1);
          Mma<T>::run(sc[2 * np + 1], qa[ks], b2, b3);
        }
      }
      // ---- scale, causal mask, online softmax ---------------------------------
      const bool need_mask = key0 + BK - 1 > pos_r0;
      float mx0 = -INFINITY, mx1 = -INFINITY;
#pragma unroll
      for (int j = 0; j < NTS; ++j) {
        const int k = key0 + 8 * j + 2 * tq;
#pragma unroll
        for (int e = 0; e < 2; ++e) {
          float x0 = sc[j][e] * a.scale_log2;
          float x1 = sc[j][2 + e] * a.scale_log2;
          if (need_mask) {
            if (k + e > pos_r0) x0 = -INFINITY;
            if (k + e > pos_r1) x1 = -INFINITY;
          }
          sc[j][e] = x0;
          sc[j][2 + e] = x1;
          mx0 = fmaxf(mx0, x0);
          mx1 = fmaxf(mx1, x1);
        }
      }
      mx0 = warp_max_xor(mx0, 1, 2);
      mx1 = warp_max_xor(mx1, 1, 2);
      const float mn0 = fmaxf(m_run[0], mx0);
      const float mn1 = fmaxf(m_run[1], mx1);
      const float mu0 = (mn0 == -INFINITY) ? 0.f : mn0;
      const float mu1 = (mn1 == -INFINITY) ? 0.f : mn1;
      const float al0 = exp2f(m_run[0] - mu0);
      const float al1 = exp2f(m_run[1] - mu1);
      m_run[0] = mn0;
      m_run[1] = mn1;
      float ls0 = 0.f, ls1 = 0.f;
#pragma unroll
      for (int j = 0; j < NTS; ++j) {
        sc[j][0] = exp2f(sc[j][0] - mu0);
        sc[j][1] = exp2f(sc[j][1] - mu0);
        sc[j][2] = exp2f(sc[j][2] - mu1);
        sc[j][3] = exp2f(sc[j][3] - mu1);
        ls0 += sc[j][0] + sc[j][1];
        ls1 += sc[j][2] + sc[j][3];
      }
      l_run[0] = l_run[0] * al0 + ls0;
      l_run[1] = l_run[1] * al1 + ls1;
#pragma unroll
      for (int j = 0; j < NTO; ++j) {
        o[j][0] *= al0;
        o[j][1] *= al0;
        o[j][2] *= al1;
        o[j][3] *= al1;
      }
      // ---- O += P V -----------------------------------------------------------
      const bool tail = key0 + BK > c;   // value rows past the context must read as zero
#pragma unroll
      for (int kk = 0; kk < BK / 16; ++kk) {
        uint32_t pa[4];
        pa[0] = Mma<T>::pack(sc[2 * kk][0], sc[2 * kk][1]);
        pa[1] = Mma<T>::pack(sc[2 * kk][2], sc[2 * kk][3]);
        pa[2] = Mma<T>::pack(sc[2 * kk + 1][0], sc[2 * kk + 1][1]);
        pa[3] = Mma<T>::pack(sc[2 * kk + 1][2], sc[2 * kk + 1][3]);
        const int kr = kk * 16 + vb_row;
        uint32_t keep_lo = 0xffffffffu, keep_hi = 0xffffffffu;
        if (tail) {
          const int k_lo = key0 + kk * 16 + 2 * tq;   // keys of b0b1
          const int k_hi = k_lo + 8;                  // keys of b2b3
          keep_lo = (k_lo < c ? 0x0000ffffu : 0u) | (k_lo + 1 < c ? 0xffff0000u : 0u);
          keep_hi = (k_hi < c ? 0x0000ffffu : 0u) | (k_hi + 1 < c ? 0xffff0000u : 0u);
        }
#pragma unroll
        for (int dp = 0; dp < NTO / 2; ++dp) {
          const int ch = 2 * dp + vb_chk;
          uint32_t b0, b1, b2, b3;
          ldsm_x4_trans(vt_s + (kr >> 4) * BLKT + (ch >> 3) * BOX + swz128(kr & 15, ch & 7), b0, b1,
                        b2, b3);
          Mma<T>::run(o[2 * dp], pa, b0 & keep_lo, b1 & keep_hi);
          Mma<T>::run(o[2 * dp + 1], pa, b2 & keep_lo, b3 & keep_hi);
        }
      }
    }
    __syncthreads();   // every warp is done with this stage
    if (threadIdx.x == 0 && kt + NS < n_kt) {
      fence_proxy_async_smem();
      issue(kt + NS);
    }
  }
  if (fail_kt >= 0) {
    // a copy never completed: record it and let the copies still in flight
    // land (bounded) before the CTA exits
    if (threadIdx.x == 0) {
      flag_status(a.status, PA_DEV_WAIT_TIMEOUT);
      const int last = min(n_kt, fail_kt + NS);
      for (int j = fail_kt; j < last; ++j)
        mbar_wait_bounded(bar0 + 8 * (j % NS), (j / NS) & 1, 100000000ull);
    }
    __syncthreads();
    return;
  }

  l_run[0] = warp_sum_xor(l_run[0], 1, 2);
  l_run[1] = warp_sum_xor(l_run[1], 1, 2);
  const float inv0 = l_run[0] > 0.f ? 1.f / l_run[0] : 0.f;
  const float inv1 = l_run[1] > 0.f ? 1.f / l_run[1] : 0.f;
  T* out = static_cast<T*>(a.out);
#pragma unroll
  for (int j = 0; j < NTO; ++j) {
    const int d = j * 8 + 2 * tq;
    if (lr0 < n)
      *reinterpret_cast<uint32_t*>(out + ((static_cast<size_t>(q0) + lr0) * a.num_q_heads + hq) * D + d) =
          Mma<T>::pack(o[j][0] * inv0, o[j][1] * inv0);
    if (lr1 < n)
      *reinterpret_cast<uint32_t*>(out + ((static_cast<size_t>(q0) + lr1) * a.num_q_heads + hq) * D + d) =
          Mma<T>::pack(o[j][2] * inv1, o[j][3] * inv1);
  }
}

namespace {
template <typename T, int D>
cudaError_t launch_prefill_t(const PrefillArgs& a, const CUtensorMap& kmap, const CUtensorMap& vmap,
                             cudaStream_t stream) {
  constexpr int NS = 2;
  constexpr int STAGE = 2 * 4 * (D / 64) * 16 * 128;
  const int smem = NS * STAGE + 1024;
  auto kern = prefill_tc_kernel<T, D, NS>;
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
  if (e != cudaSuccess) return e;
  dim3 grid((a.max_q_len + 63) / 64, a.num_q_heads, a.num_seqs);
  return launch_pdl(kern, grid, dim3(128), smem, stream, kmap, vmap, a);
}
}  // namespace

cudaError_t launch_prefill_tc(const PrefillArgs& a, int dtype, const CUtensorMap& kmap,
                              const CUtensorMap& vmap, cudaStream_t stream) {
  if (dtype == PA_BF16) {
    return a.head_dim == 128 ? launch_prefill_t<__nv_bfloat16, 128>(a, kmap, vmap, stream)
                             : launch_prefill_t<__nv_bfloat16, 64>(a, kmap, vmap, stream);
  }
  return a.head_dim == 128 ? launch_prefill_t<__half, 128>(a, kmap, vmap, stream)
                           : launch_prefill_t<__half, 64>(a, kmap, vmap, stream);
}

}  // namespace pa
