// decode_tc.cu -- paged decode attention on the tensor cores (bf16 / fp16).
//
// One query token per sequence against its whole paged cache, grouped-query
// heads sharing each KV head ("LLM Inference Server From Scratch", How it
// works, 4 Attention Kernel: GQA; "LLM Inference Server", Stage 1: decode
// passes only the new token).  Decode is bound by HBM bandwidth ("LLM
// Inference Server", What You Will Build), so the kernel is organised around
// moving every K/V byte exactly once:
//
//  * grid = (split, kv head, sequence).  A CTA owns one partition of
//    part_blocks pool blocks of one (sequence, KV head), and all G query heads
//    of that group, so each K/V tile is read from HBM once for the whole group.
//  * W warps per CTA; warp w takes the partition's blocks w, w+W, ... and runs
//    its own NS-stage TMA pipeline: lane 0 issues 2-D tensor copies of the
//    (block, head) K and V tiles (16 x D, 128-byte swizzled) into shared
//    memory, completing on a per-stage mbarrier.  No CTA-wide barrier in the
//    main loop.
//  * Per 16-token block: S^T = K q^T with mma.sync m16n8k16 (tokens = M,
//    query heads of the group = N padded to 8, head dim = K), fp32 online
//    softmax in the log2 domain (scale folded with log2 e), P^T moved into the
//    B-operand layout with movmatrix, and O^T += V^T P^T with V read through
//    ldmatrix.trans.  Accumulators stay in registers.
//  * The softmax reference is raised lazily: a warp vote finds the blocks
//    with a score more than 2^8 above it, and only those pay for the
//    cross-lane maximum and the rescale of the accumulators; the weights of
//    every other block are exponentials against the current reference (<= 256,
//    exact in the final normalisation).
//  * The W warp states are merged in shared memory; the CTA writes the final
//    row (one partition) or a normalised partial plus its log2-sum-exp2; the
//    last partition of a (sequence, KV head) to finish merges them all by
//    log-sum-exp (see decode_merge.cuh).
//
// The last block of a sequence is partial: scores of positions past the
// context are set to -inf and the matching V elements are zeroed, so stale
// pool contents (even NaN/Inf) never leak into the result.
#include "decode_merge.cuh"
#include "pa_common.cuh"
#include "pa_internal.h"

namespace pa {

namespace {
constexpr float kLazy = 8.f;   // log2 headroom of the softmax reference
}

template <typename T, int D, int W, int NS>
__global__ void __launch_bounds__(W * 32)
decode_tc_kernel(const __grid_constant__ CUtensorMap kmap, const __grid_constant__ CUtensorMap vmap,
                 const DecodeArgs a) {
  constexpr int NBOX = D / 64;         // 64-element (128-byte) TMA boxes per tile row
  constexpr int BOX = 16 * 128;        // one box: 16 tokens x 128 bytes
  constexpr int TILE = NBOX * BOX;     // one (block, head) tile of K or V
  constexpr int STAGE = 2 * TILE;      // K tile then V tile
  constexpr int KS = D / 16;           // k-steps of the score MMA / m-tiles of the PV MMA

  extern __shared__ uint8_t smem_raw[];
  __shared__ __align__(8) uint64_t bars[W * NS];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                             ~static_cast<uintptr_t>(1023));

  const int split = blockIdx.x;
  const int kvh = blockIdx.y;
  const int s = blockIdx.z;
  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const int G = a.num_q_heads / a.num_kv_heads;

  grid_dependency_wait();   // inputs may come from the kernel just before us
  if (threadIdx.x == 0) {
    prefetch_tensormap(&kmap);
    prefetch_tensormap(&vmap);
  }
  // This warp's block-table entries of the partition (warp w takes blocks w,
  // w + W, ...), one per lane, loaded before the context length is known so
  // that the two loads overlap: entries below max_blocks_per_seq always exist.
  const int blk0 = split * a.part_blocks;
  const int jl = warp + lane * W;   // partition-local block of this lane
  int my_id = 0;
  if (jl < a.part_blocks && blk0 + jl < a.max_blocks_per_seq)
    my_id = __ldg(a.block_tables + static_cast<size_t>(s) * a.max_blocks_per_seq + blk0 + jl);
  // Decode step with the append fused in: this sequence's new K and V rows of
  // this KV head, 16 bytes per lane (K in lanes 0..CH-1, V in CH..2CH-1).
  constexpr int CH = D * static_cast<int>(sizeof(T)) / 16;
  uint4 new_row = make_uint4(0u, 0u, 0u, 0u);
  if (a.k_new != nullptr && lane < 2 * CH) {
    const bool is_v = lane >= CH;
    new_row = __ldg(static_cast<const uint4*>(is_v ? a.v_new : a.k_new) +
                    (static_cast<size_t>(s) * a.num_kv_heads + kvh) * CH + (is_v ? lane - CH : lane));
  }
  const int ctx = checked_context(a, s, threadIdx.x == 0 && split == 0 && kvh == 0);
  const int nblk_seq = (ctx + kBlock - 1) / kBlock;
  const int n_splits = (nblk_seq + a.part_blocks - 1) / a.part_blocks;
  if (ctx == 0) {
    if (split == 0) store_zero_rows<T, D>(a, G, s, kvh, W * 32);
    return;
  }
  if (split >= n_splits) return;
  const int nblk = min(a.part_blocks, nblk_seq - blk0);
  const int nb_w = nblk > warp ? (nblk - warp + W - 1) / W : 0;   // <= 32 (host limit)

  // Out-of-range ids are replaced by block 0 and their tokens masked out.
  bool my_bad = false;
  if (lane < nb_w) {
    if (my_id < 0 || my_id >= a.num_blocks) {
      my_bad = true;
      my_id = 0;
      flag_status(a.status, PA_DEV_BAD_BLOCK_ID);
    }
  } else {
    my_id = 0;
  }
  const unsigned bad_mask = __ballot_sync(0xffffffffu, my_bad);

  if (a.k_new != nullptr && split == n_splits - 1 && warp == (nblk - 1) % W) {
    // The new token (position ctx - 1) lies in the sequence's last block, which
    // this warp reads: write it, then order the writes before the warp's own
    // TMA copies (async proxy) of that block.
    const int li = (nblk - 1) / W;   // lane holding the block's id
    const int id = __shfl_sync(0xffffffffu, my_id, li);
    if (!((bad_mask >> li) & 1u) && lane < 2 * CH) {
      const size_t row = (static_cast<size_t>(id) * a.num_kv_heads + kvh) * kBlock + (ctx - 1) % kBlock;
      const bool is_v = lane >= CH;
      uint4* pool = static_cast<uint4*>(const_cast<void*>(is_v ? a.v_pool : a.k_pool));
      pool[row * CH + (is_v ? lane - CH : lane)] = new_row;
    }
    asm volatile("fence.proxy.async.global;" ::: "memory");
    __syncwarp();
  }

  const uint32_t wbase = smem_u32(smem + warp * NS * STAGE);
  const uint32_t bar0 = smem_u32(&bars[warp * NS]);
  const uint64_t policy = l2_policy_evict_first();
  if (lane == 0) {
    for (int st = 0; st < NS; ++st) mbar_init(bar0 + 8 * st, 1);
    fence_barrier_init();
  }
  __syncwarp();

  // Issue the K and V tiles of this warp's i-th block into stage i % NS.
  auto issue = [&](int i) {
    const int id = __shfl_sync(0xffffffffu, my_id, i);
    if (lane == 0) {
      const int st = i % NS;
      const uint32_t bar = bar0 + 8 * st;
      const uint32_t dst = wbase + st * STAGE;
      const int y = (id * a.num_kv_heads + kvh) * kBlock;
      mbar_arrive_expect_tx(bar, STAGE);
#pragma unroll
      for (int b = 0; b < NBOX; ++b) {
        tma_load_2d(dst + b * BOX, &kmap, b * 64, y, bar, policy);
        tma_load_2d(dst + TILE + b * BOX, &vmap, b * 64, y, bar, policy);
      }
    }
  };
  const int npro = nb_w < NS ? nb_w : NS;
  for (int i = 0; i < npro; ++i) issue(i);

  // Query fragments: B operand (k = head dim, n = query head of the group).
  const int g = lane >> 2;   // fragment row group
  const int tq = lane & 3;   // thread in group
  uint32_t qf[KS][2];
  {
    const T* qrow = static_cast<const T*>(a.q) +
                    (static_cast<size_t>(s) * a.num_q_heads + kvh * G + (g < G ? g : 0)) * D;
#pragma unroll
    for (int ks = 0; ks < KS; ++ks) {
      if (g < G) {
        qf[ks][0] = *reinterpret_cast<const uint32_t*>(qrow + ks * 16 + 2 * tq);
        qf[ks][1] = *reinterpret_cast<const uint32_t*>(qrow + ks * 16 + 8 + 2 * tq);
      } else {
        qf[ks][0] = 0u;
        qf[ks][1] = 0u;
      }
    }
  }

  // Online-softmax state for query heads 2*tq and 2*tq+1 (log2 domain).  The
  // reference m_ref is raised lazily: only when a score exceeds it by more than
  // kLazy, so unnormalised weights stay <= 2^kLazy and most blocks need no
  // cross-lane reduction and no rescale of the accumulators.
  float m_ref[2] = {-INFINITY, -INFINITY};
  float mu[2] = {0.f, 0.f};   // m_ref, or 0 while it is -inf
  float l_run[2] = {0.f, 0.f};
  float acc[KS][4];
#pragma unroll
  for (int mt = 0; mt < KS; ++mt) acc[mt][0] = acc[mt][1] = acc[mt][2] = acc[mt][3] = 0.f;

  // ldmatrix row/chunk owned by this lane (see the fragment layouts of m16n8k16)
  const int k_row = (lane & 7) + ((lane >> 3) & 1) * 8;   // K as A: token row
  const int k_chk = lane >> 4;                            //          +0/+1 chunk
  const int v_row = (lane & 7) + (lane >> 4) * 8;         // V^T via .trans: token row
  const int v_chk = (lane >> 3) & 1;                      //          +0/+1 chunk

  bool ok = true;
  int i = 0;
  for (; i < nb_w; ++i) {
    const int st = i % NS;
    const bool got = mbar_wait_bounded(bar0 + 8 * st, (i / NS) & 1);
    if (!__all_sync(0xffffffffu, got)) {
      ok = false;
      break;
    }
    const uint32_t kt = wbase + st * STAGE;
    const uint32_t vt = kt + TILE;
    const int lb = blk0 + warp + i * W;
    int nvalid = ctx - lb * kBlock;
    nvalid = nvalid > kBlock ? kBlock : nvalid;
    if (bad_mask & (1u << i)) nvalid = 0;

    // ---- scores: S^T[token][head] = K[token] . q[head] -------------------
    float sa[4] = {0.f, 0.f, 0.f, 0.f};
    float sb[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
    for (int ks = 0; ks < KS; ++ks) {
      const int ch = 2 * ks + k_chk;
      uint32_t af[4];
      ldsm_x4(kt + (ch >> 3) * BOX + swz128(k_row, ch & 7), af[0], af[1], af[2], af[3]);
      if (ks & 1)
        Mma<T>::run(sb, af, qf[ks][0], qf[ks][1]);
      else
        Mma<T>::run(sa, af, qf[ks][0], qf[ks][1]);
    }
    // sa[0], sa[1]: token g, heads 2tq, 2tq+1; sa[2], sa[3]: token g+8
    float x0 = (g < nvalid) ? (sa[0] + sb[0]) * a.scale_log2 : -INFINITY;
    float x1 = (g < nvalid) ? (sa[1] + sb[1]) * a.scale_log2 : -INFINITY;
    float x2 = (g + 8 < nvalid) ? (sa[2] + sb[2]) * a.scale_log2 : -INFINITY;
    float x3 = (g + 8 < nvalid) ? (sa[3] + sb[3]) * a.scale_log2 : -INFINITY;

    // ---- raise the reference (rare) -------------------------------------------
    const bool grow = fmaxf(x0, x2) > m_ref[0] + kLazy || fmaxf(x1, x3) > m_ref[1] + kLazy;
    if (__any_sync(0xffffffffu, grow)) {
      const float mb0 = warp_max_xor(fmaxf(x0, x2), 4, 16);
      const float mb1 = warp_max_xor(fmaxf(x1, x3), 4, 16);
      const float mn0 = fmaxf(m_ref[0], mb0);
      const float mn1 = fmaxf(m_ref[1], mb1);
      const float nu0 = mn0 == -INFINITY ? 0.f : mn0;
      const float nu1 = mn1 == -INFINITY ? 0.f : mn1;
      const float al0 = fast_exp2(m_ref[0] - nu0);
      const float al1 = fast_exp2(m_ref[1] - nu1);
      l_run[0] *= al0;
      l_run[1] *= al1;
#pragma unroll
      for (int mt = 0; mt < KS; ++mt) {
        acc[mt][0] *= al0;
        acc[mt][1] *= al1;
        acc[mt][2] *= al0;
        acc[mt][3] *= al1;
      }
      m_ref[0] = mn0;
      m_ref[1] = mn1;
      mu[0] = nu0;
      mu[1] = nu1;
    }
    // The weights enter the PV product rounded to T; the normaliser sums the
    // same rounded values, so numerator and denominator use identical weights.
    const uint32_t pk0 = Mma<T>::pack(fast_exp2(x0 - mu[0]), fast_exp2(x1 - mu[1]));   // token g
    const uint32_t pk1 = Mma<T>::pack(fast_exp2(x2 - mu[0]), fast_exp2(x3 - mu[1]));   // token g + 8
    const float2 r0 = Mma<T>::unpack(pk0);
    const float2 r1 = Mma<T>::unpack(pk1);
    l_run[0] += r0.x + r1.x;
    l_run[1] += r0.y + r1.y;

    // P^T as the B operand (k = token, n = head): transpose the two 8x8 halves
    const uint32_t pb0 = movmatrix_trans(pk0);
    const uint32_t pb1 = movmatrix_trans(pk1);

    // ---- O^T[d][head] += V^T[d][token] P^T[token][head] --------------------
    const bool partial = nvalid < kBlock;
#pragma unroll
    for (int mt = 0; mt < KS; ++mt) {
      const int ch = 2 * mt + v_chk;
      uint32_t vf[4];
      ldsm_x4_trans(vt + (ch >> 3) * BOX + swz128(v_row, ch & 7), vf[0], vf[1], vf[2], vf[3]);
      if (partial) {
        // vf[0], vf[1] hold tokens 2tq, 2tq+1; vf[2], vf[3] tokens 2tq+8, 2tq+9
        const uint32_t lo0 = (2 * tq < nvalid) ? 0x0000ffffu : 0u;
        const uint32_t hi0 = (2 * tq + 1 < nvalid) ? 0xffff0000u : 0u;
        const uint32_t lo1 = (2 * tq + 8 < nvalid) ? 0x0000ffffu : 0u;
        const uint32_t hi1 = (2 * tq + 9 < nvalid) ? 0xffff0000u : 0u;
        vf[0] &= lo0 | hi0;
        vf[1] &= lo0 | hi0;
        vf[2] &= lo1 | hi1;
        vf[3] &= lo1 | hi1;
      }
      Mma<T>::run(acc[mt], vf, pb0, pb1);
    }

    // the stage is free once every lane's ldmatrix has completed
    __syncwarp();
    if (i + NS < nb_w) {
      fence_proxy_async_smem();
      issue(i + NS);
    }
  }

  if (!ok) {
    if (lane == 0) flag_status(a.status, PA_DEV_WAIT_TIMEOUT);
    // let copies still in flight land (bounded) before the CTA can exit
    const int last = (i + NS < nb_w) ? i + NS : nb_w;
    for (int j = i; j < last; ++j) mbar_wait_bounded(bar0 + 8 * (j % NS), (j / NS) & 1, 100000000ull);
  }

  // the per-lane partial sums of p cover the lane's own tokens: reduce over g
  l_run[0] = warp_sum_xor(l_run[0], 4, 16);
  l_run[1] = warp_sum_xor(l_run[1], 4, 16);

  // ---- merge the W warp states through shared memory -------------------------
  __syncthreads();
  float* red_o = reinterpret_cast<float*>(smem);
  float* red_m = red_o + W * 8 * D;
  float* red_l = red_m + W * 8;
  const int h0 = 2 * tq;
  const int h1 = 2 * tq + 1;
#pragma unroll
  for (int mt = 0; mt < KS; ++mt) {
    const int d0 = mt * 16 + g;
    if (h0 < G) {
      red_o[(warp * 8 + h0) * D + d0] = acc[mt][0];
      red_o[(warp * 8 + h0) * D + d0 + 8] = acc[mt][2];
    }
    if (h1 < G) {
      red_o[(warp * 8 + h1) * D + d0] = acc[mt][1];
      red_o[(warp * 8 + h1) * D + d0 + 8] = acc[mt][3];
    }
  }
  if (g == 0) {
    if (h0 < G) {
      red_m[warp * 8 + h0] = m_ref[0];
      red_l[warp * 8 + h0] = l_run[0];
    }
    if (h1 < G) {
      red_m[warp * 8 + h1] = m_ref[1];
      red_l[warp * 8 + h1] = l_run[1];
    }
  }
  __syncthreads();
  cta_merge_store<T, W, D>(a, red_o, red_m, red_l, G, s, kvh, split, n_splits);
}

namespace {

template <typename T, int D, int NS>
cudaError_t launch_tc_ns(const DecodeArgs& a, const CUtensorMap& kmap, const CUtensorMap& vmap,
                         cudaStream_t stream) {
  constexpr int W = 4;
  constexpr int STAGE = 2 * (D / 64) * 16 * 128;
  static_assert(W * 8 * D * 4 + W * 16 * 4 <= W * NS * STAGE, "merge buffer must fit");
  const int smem = W * NS * STAGE + 1024;
  auto kern = decode_tc_kernel<T, D, W, NS>;
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
  if (e != cudaSuccess) return e;
  dim3 grid(a.max_splits, a.num_kv_heads, a.num_seqs);
  return launch_pdl(kern, grid, dim3(W * 32), smem, stream, kmap, vmap, a);
}

// Stages per warp: 64 KB of stages per CTA fits three CTAs on an SM (192 KB in
// flight per SM).  When the grid has fewer CTAs than that per SM, each CTA
// takes the stages the absent ones would have used (96 or 192 KB), so that
// small batches keep as many bytes in flight per SM as large ones.
template <typename T, int D>
cudaError_t launch_tc_t(const DecodeArgs& a, const CUtensorMap& kmap, const CUtensorMap& vmap,
                        cudaStream_t stream) {
  constexpr int NS1 = (D == 128) ? 2 : 4;   // 16 KB per warp
  int sms = device_sm_count();
  if (sms <= 0) sms = 152;
  const long long ctas = static_cast<long long>(a.max_splits) * a.num_kv_heads * a.num_seqs;
  if (ctas <= sms) return launch_tc_ns<T, D, 3 * NS1>(a, kmap, vmap, stream);
  if (ctas <= 2LL * sms) return launch_tc_ns<T, D, 3 * NS1 / 2>(a, kmap, vmap, stream);
  return launch_tc_ns<T, D, NS1>(a, kmap, vmap, stream);
}

}  // namespace

cudaError_t launch_decode_tc(const DecodeArgs& a, int dtype, const CUtensorMap& kmap,
                             const CUtensorMap& vmap, cudaStream_t stream) {
  if (dtype == PA_BF16) {
    return a.head_dim == 128 ? launch_tc_t<__nv_bfloat16, 128>(a, kmap, vmap, stream)
                             : launch_tc_t<__nv_bfloat16, 64>(a, kmap, vmap, stream);
  }
  return a.head_dim == 128 ? launch_tc_t<__half, 128>(a, kmap, vmap, stream)
                           : launch_tc_t<__half, 64>(a, kmap, vmap, stream);
}

}  // namespace pa
