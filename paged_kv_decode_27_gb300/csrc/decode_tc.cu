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

// NT = 8-column tiles of query columns (MMA N): 1 for decode (the G query
// heads of the group, padded to 8), up to 4 to verify drafted tokens (G heads
// at each of q_len positions, column c = i * G + h).  With NT > 1 the q rows
// live in shared memory and the B fragments are read with ldmatrix each
// block; with NT = 1 they stay in registers.
template <typename T, int D, int W, int NS, int NT>
__global__ void __launch_bounds__(W * 32)
decode_tc_kernel(const __grid_constant__ CUtensorMap kmap, const __grid_constant__ CUtensorMap vmap,
                 const DecodeArgs a) {
  constexpr int NBOX = D / 64;         // 64-element (128-byte) TMA boxes per tile row
  constexpr int BOX = 16 * 128;        // one box: 16 tokens x 128 bytes
  constexpr int TILE = NBOX * BOX;     // one (block, head) tile of K or V
  constexpr int STAGE = 2 * TILE;      // K tile then V tile
  constexpr int KS = D / 16;           // k-steps of the score MMA / m-tiles of the PV MMA
  constexpr int NC = 8 * NT;           // query columns per warp in the merge buffers
  constexpr int QROW = D * 2 + 16;     // padded shared-memory row of q (NT > 1)

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
  const int NQ = G * a.q_len;          // query columns of this (sequence, KV head), <= NC

  grid_dependency_wait();   // inputs may come from the kernel just before us
  const int ctx = checked_context(a, s, threadIdx.x == 0 && split == 0 && kvh == 0);
  const int nblk_seq = (ctx + kBlock - 1) / kBlock;
  const int n_splits = (nblk_seq + a.part_blocks - 1) / a.part_blocks;
  if (ctx == 0) {
    if (split == 0) store_zero_rows<T, D>(a, G, s, kvh, W * 32);
    return;
  }
  if (split >= n_splits) return;
  const int blk0 = split * a.part_blocks;
  const int nblk = min(a.part_blocks, nblk_seq - blk0);
  const int nb_w = nblk > warp ? (nblk - warp + W - 1) / W : 0;   // <= 32 (host limit)

  // Physical ids of this warp's blocks, one per lane; out-of-range ids are
  // replaced by block 0 and their tokens masked out.
  int my_id = 0;
  bool my_bad = false;
  if (lane < nb_w) {
    int id = __ldg(a.block_tables + static_cast<size_t>(s) * a.max_blocks_per_seq + blk0 + warp +
                   lane * W);
    if (id < 0 || id >= a.num_blocks) {
      my_bad = true;
      id = 0;
      flag_status(a.status, PA_DEV_BAD_BLOCK_ID);
    }
    my_id = id;
  }
  const unsigned bad_mask = __ballot_sync(0xffffffffu, my_bad);

  const uint32_t wbase = smem_u32(smem + warp * NS * STAGE);
  const uint32_t bar0 = smem_u32(&bars[warp * NS]);
  const uint64_t policy = l2_policy_evict_first();
  if (lane == 0) {
    for (int st = 0; st < NS; ++st) mbar_init(bar0 + 8 * st, 1);
    fence_barrier_init();
    prefetch_tensormap(&kmap);
    prefetch_tensormap(&vmap);
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

  const int g = lane >> 2;   // fragment row group
  const int tq = lane & 3;   // thread in group

  // Query fragments: B operand (k = head dim, n = query column), in registers
  // for NT = 1, else as padded rows in shared memory behind the stages.
  uint32_t qf[NT == 1 ? KS : 1][2];
  const uint32_t qs = smem_u32(smem + W * NS * STAGE);   // q rows (NT > 1)
  if constexpr (NT == 1) {
    const T* qrow = static_cast<const T*>(a.q) + query_row(a, s, kvh, G, g < NQ ? g : 0) * D;
#pragma unroll
    for (int ks = 0; ks < KS; ++ks) {
      if (g < NQ) {
        qf[ks][0] = *reinterpret_cast<const uint32_t*>(qrow + ks * 16 + 2 * tq);
        qf[ks][1] = *reinterpret_cast<const uint32_t*>(qrow + ks * 16 + 8 + 2 * tq);
      } else {
        qf[ks][0] = 0u;
        qf[ks][1] = 0u;
      }
    }
  } else {
    // the CTA's NC query rows (zero past NQ), 16 bytes per thread per step
    uint8_t* qdst = smem + W * NS * STAGE;
    for (int idx = threadIdx.x; idx < NC * (D / 8); idx += W * 32) {
      const int n = idx / (D / 8);
      const int chunk = idx - n * (D / 8);
      uint4 v = make_uint4(0u, 0u, 0u, 0u);
      if (n < NQ)
        v = *reinterpret_cast<const uint4*>(static_cast<const T*>(a.q) + query_row(a, s, kvh, G, n) * D +
                                            chunk * 8);
      *reinterpret_cast<uint4*>(qdst + n * QROW + chunk * 16) = v;
    }
    __syncthreads();
  }
  // ldmatrix of the 32-column k slice of a pair of k-steps: lane l addresses
  // row (l & 7) of matrix l >> 3 = (step of the pair, low / high 8 columns)
  const uint32_t q_lane = qs + (lane & 7) * QROW + ((lane >> 3) * 8) * 2;

  // Causal limit of this lane's score columns n = 8t + 2tq + e: query
  // position i = n / G of the sequence sits at ctx - q_len + i and sees keys up
  // to it (for decode, q_len = 1: every cached key).
  int lim[NT][2];
#pragma unroll
  for (int t = 0; t < NT; ++t) {
#pragma unroll
    for (int e = 0; e < 2; ++e) {
      const int n = 8 * t + 2 * tq + e;
      lim[t][e] = n < NQ ? ctx - a.q_len + n / G : ctx - 1;
    }
  }

  // Online-softmax state of this lane's columns (log2 domain).  The reference
  // m_ref is raised lazily: only when a score exceeds it by more than kLazy,
  // so unnormalised weights stay <= 2^kLazy and most blocks need no
  // cross-lane reduction and no rescale of the accumulators.
  float m_ref[NT][2], mu[NT][2], l_run[NT][2];
  float acc[KS][NT][4];
#pragma unroll
  for (int t = 0; t < NT; ++t) {
    m_ref[t][0] = m_ref[t][1] = -INFINITY;
    mu[t][0] = mu[t][1] = 0.f;   // m_ref, or 0 while it is -inf
    l_run[t][0] = l_run[t][1] = 0.f;
#pragma unroll
    for (int mt = 0; mt < KS; ++mt) acc[mt][t][0] = acc[mt][t][1] = acc[mt][t][2] = acc[mt][t][3] = 0.f;
  }

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

    // ---- scores: S^T[token][column] = K[token] . q[column] -----------------
    float sa[NT][4], sb[NT][4];
#pragma unroll
    for (int t = 0; t < NT; ++t) {
      sa[t][0] = sa[t][1] = sa[t][2] = sa[t][3] = 0.f;
      sb[t][0] = sb[t][1] = sb[t][2] = sb[t][3] = 0.f;
    }
#pragma unroll
    for (int kp = 0; kp < KS / 2; ++kp) {   // pairs of k-steps
      uint32_t ae[4], ao[4];
      const int ce = 4 * kp + k_chk, co = ce + 2;
      ldsm_x4(kt + (ce >> 3) * BOX + swz128(k_row, ce & 7), ae[0], ae[1], ae[2], ae[3]);
      ldsm_x4(kt + (co >> 3) * BOX + swz128(k_row, co & 7), ao[0], ao[1], ao[2], ao[3]);
#pragma unroll
      for (int t = 0; t < NT; ++t) {
        if constexpr (NT == 1) {
          Mma<T>::run(sa[t], ae, qf[2 * kp][0], qf[2 * kp][1]);
          Mma<T>::run(sb[t], ao, qf[2 * kp + 1][0], qf[2 * kp + 1][1]);
        } else {
          // one ldmatrix.x4 holds the B fragments of both k-steps of the pair
          uint32_t r0, r1, r2, r3;
          ldsm_x4(q_lane + (8 * t) * QROW + kp * 64, r0, r1, r2, r3);
          Mma<T>::run(sa[t], ae, r0, r1);
          Mma<T>::run(sb[t], ao, r2, r3);
        }
      }
    }
    // [t][0], [t][1]: token g, columns 8t+2tq, +1; [t][2], [t][3]: token g+8
    const int kp0 = lb * kBlock + g, kp1 = kp0 + 8;
    const bool in0 = g < nvalid, in1 = g + 8 < nvalid;
    float x[NT][4];
    bool grow = false;
#pragma unroll
    for (int t = 0; t < NT; ++t) {
      x[t][0] = (in0 && kp0 <= lim[t][0]) ? (sa[t][0] + sb[t][0]) * a.scale_log2 : -INFINITY;
      x[t][1] = (in0 && kp0 <= lim[t][1]) ? (sa[t][1] + sb[t][1]) * a.scale_log2 : -INFINITY;
      x[t][2] = (in1 && kp1 <= lim[t][0]) ? (sa[t][2] + sb[t][2]) * a.scale_log2 : -INFINITY;
      x[t][3] = (in1 && kp1 <= lim[t][1]) ? (sa[t][3] + sb[t][3]) * a.scale_log2 : -INFINITY;
      grow = grow || fmaxf(x[t][0], x[t][2]) > m_ref[t][0] + kLazy ||
             fmaxf(x[t][1], x[t][3]) > m_ref[t][1] + kLazy;
    }

    // ---- raise the references (rare) -------------------------------------------
    if (__any_sync(0xffffffffu, grow)) {
#pragma unroll
      for (int t = 0; t < NT; ++t) {
#pragma unroll
        for (int e = 0; e < 2; ++e) {
          const float mb = warp_max_xor(fmaxf(x[t][e], x[t][e + 2]), 4, 16);
          const float mn = fmaxf(m_ref[t][e], mb);
          const float nu = mn == -INFINITY ? 0.f : mn;
          const float al = fast_exp2(m_ref[t][e] - nu);
          l_run[t][e] *= al;
#pragma unroll
          for (int mt = 0; mt < KS; ++mt) {
            acc[mt][t][e] *= al;
            acc[mt][t][e + 2] *= al;
          }
          m_ref[t][e] = mn;
          mu[t][e] = nu;
        }
      }
    }
    uint32_t pb[NT][2];
#pragma unroll
    for (int t = 0; t < NT; ++t) {
      const float p0 = fast_exp2(x[t][0] - mu[t][0]);
      const float p1 = fast_exp2(x[t][1] - mu[t][1]);
      const float p2 = fast_exp2(x[t][2] - mu[t][0]);
      const float p3 = fast_exp2(x[t][3] - mu[t][1]);
      l_run[t][0] += p0 + p2;
      l_run[t][1] += p1 + p3;
      // P^T as the B operand (k = token, n = column): transpose the two 8x8 halves
      pb[t][0] = movmatrix_trans(Mma<T>::pack(p0, p1));
      pb[t][1] = movmatrix_trans(Mma<T>::pack(p2, p3));
    }

    // ---- O^T[d][column] += V^T[d][token] P^T[token][column] ---------------------
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
#pragma unroll
      for (int t = 0; t < NT; ++t) Mma<T>::run(acc[mt][t], vf, pb[t][0], pb[t][1]);
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
#pragma unroll
  for (int t = 0; t < NT; ++t) {
    l_run[t][0] = warp_sum_xor(l_run[t][0], 4, 16);
    l_run[t][1] = warp_sum_xor(l_run[t][1], 4, 16);
  }

  // ---- merge the W warp states through shared memory -------------------------
  __syncthreads();
  float* red_o = reinterpret_cast<float*>(smem);
  float* red_m = red_o + W * NC * D;
  float* red_l = red_m + W * NC;
#pragma unroll
  for (int t = 0; t < NT; ++t) {
    const int n0 = 8 * t + 2 * tq;
    const int n1 = n0 + 1;
#pragma unroll
    for (int mt = 0; mt < KS; ++mt) {
      const int d0 = mt * 16 + g;
      if (n0 < NQ) {
        red_o[(warp * NC + n0) * D + d0] = acc[mt][t][0];
        red_o[(warp * NC + n0) * D + d0 + 8] = acc[mt][t][2];
      }
      if (n1 < NQ) {
        red_o[(warp * NC + n1) * D + d0] = acc[mt][t][1];
        red_o[(warp * NC + n1) * D + d0 + 8] = acc[mt][t][3];
      }
    }
    if (g == 0) {
      if (n0 < NQ) {
        red_m[warp * NC + n0] = m_ref[t][0];
        red_l[warp * NC + n0] = l_run[t][0];
      }
      if (n1 < NQ) {
        red_m[warp * NC + n1] = m_ref[t][1];
        red_l[warp * NC + n1] = l_run[t][1];
      }
    }
  }
  __syncthreads();
  cta_merge_store<T, W, D, NC>(a, red_o, red_m, red_l, G, s, kvh, split, n_splits);
}

namespace {

template <typename T, int D, int NT>
cudaError_t launch_tc_t(const DecodeArgs& a, const CUtensorMap& kmap, const CUtensorMap& vmap,
                        cudaStream_t stream) {
  constexpr int W = 4;
  // 64 KB of stages and 3 CTAs per SM; the widest query tiles need more
  // registers (2 CTAs per SM at D = 128), so they take deeper pipelines
  constexpr int NS = (D == 128) ? (NT >= 3 ? 3 : 2) : 4;
  constexpr int STAGE = 2 * (D / 64) * 16 * 128;
  constexpr int STAGES = W * NS * STAGE;
  constexpr int MERGE = W * 8 * NT * D * 4 + 2 * W * 8 * NT * 4;
  constexpr int QBUF = NT > 1 ? 8 * NT * (D * 2 + 16) : 0;
  const int smem = (STAGES > MERGE ? STAGES : MERGE) + QBUF + 1024;
  auto kern = decode_tc_kernel<T, D, W, NS, NT>;
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
  if (e != cudaSuccess) return e;
  dim3 grid(a.max_splits, a.num_kv_heads, a.num_seqs);
  return launch_pdl(kern, grid, dim3(W * 32), smem, stream, kmap, vmap, a);
}

template <typename T, int D>
cudaError_t launch_nt(const DecodeArgs& a, const CUtensorMap& kmap, const CUtensorMap& vmap,
                      cudaStream_t stream) {
  const int cols = (a.num_q_heads / a.num_kv_heads) * a.q_len;
  if (cols <= 8) return launch_tc_t<T, D, 1>(a, kmap, vmap, stream);
  if (cols <= 16) return launch_tc_t<T, D, 2>(a, kmap, vmap, stream);
  if (cols <= 24) return launch_tc_t<T, D, 3>(a, kmap, vmap, stream);
  return launch_tc_t<T, D, 4>(a, kmap, vmap, stream);
}

}  // namespace

cudaError_t launch_decode_tc(const DecodeArgs& a, int dtype, const CUtensorMap& kmap,
                             const CUtensorMap& vmap, cudaStream_t stream) {
  if (dtype == PA_BF16) {
    return a.head_dim == 128 ? launch_nt<__nv_bfloat16, 128>(a, kmap, vmap, stream)
                             : launch_nt<__nv_bfloat16, 64>(a, kmap, vmap, stream);
  }
  return a.head_dim == 128 ? launch_nt<__half, 128>(a, kmap, vmap, stream)
                           : launch_nt<__half, 64>(a, kmap, vmap, stream);
}

}  // namespace pa
