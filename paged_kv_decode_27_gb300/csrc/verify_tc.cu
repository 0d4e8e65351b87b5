// verify_tc.cu -- attention for the verification pass of speculative
// decoding: q_len query positions per sequence, causal over the paged cache.
//
// The target model checks K drafted tokens in one forward pass ("LLM
// Inference Server", Batched Scheduling & Speculative Decoding: K = 4), so
// each sequence has q_len = K + 1 queries; query i sits at position
// context - q_len + i and sees the keys up to it.  Per KV head the query
// columns are the G heads of the group at every position (c = i * G + h), up
// to 32 of them.
//
// All columns of a (sequence, KV head, partition) unit read the same K/V
// tiles, so the CTA streams each tile once into a ring of shared-memory
// stages and lets one consumer warp per 8-column tile read it:
//  * warp NT (producer) issues the TMA copies of block i into stage i % NS
//    once every consumer has released that stage (an "empty" mbarrier with
//    NT arrivals) and arms the stage's "full" mbarrier with the byte count;
//  * warps 0..BG*NT-1 (consumers) form BG block groups of NT warps: group b
//    takes blocks b, b+BG, ..., and warp t of a group owns 8 query columns:
//    q fragments in registers, S^T = K q^T and O^T += V^T P^T with mma.sync
//    m16n8k16 exactly as in decode, the causal limit per column, and the
//    lazily raised softmax reference; after a block the warp arrives on the
//    stage's empty barrier.
// A consumer's state is a decode warp's (under 100 registers), where one
// warp holding all 24 columns of a block would need 210 registers and half
// the occupancy; the block groups keep several blocks in flight per CTA.
// The BG warps that own a column merge through shared memory; split-K
// partials are merged by log-sum-exp as in decode.
#include "decode_merge.cuh"
#include "pa_common.cuh"
#include "pa_internal.h"

namespace pa {

namespace {
constexpr float kLazyV = 8.f;   // log2 headroom of the softmax reference
}

template <typename T, int D, int NT, int BG, int NS>
__global__ void __launch_bounds__((BG * NT + 1) * 32, (BG * NT + 1) <= 5 ? 4 : 3)
verify_tc_kernel(const __grid_constant__ CUtensorMap kmap, const __grid_constant__ CUtensorMap vmap,
                 const DecodeArgs a) {
  constexpr int NBOX = D / 64;
  constexpr int BOX = 16 * 128;
  constexpr int TILE = NBOX * BOX;
  constexpr int STAGE = 2 * TILE;
  constexpr int KS = D / 16;
  constexpr int NC = 8 * NT;
  constexpr int THREADS = (BG * NT + 1) * 32;
  constexpr int PRODUCER = BG * NT;

  extern __shared__ uint8_t smem_raw[];
  __shared__ __align__(8) uint64_t full_bar[NS];
  __shared__ __align__(8) uint64_t empty_bar[NS];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                             ~static_cast<uintptr_t>(1023));

  const int split = blockIdx.x;
  const int kvh = blockIdx.y;
  const int s = blockIdx.z;
  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const int G = a.num_q_heads / a.num_kv_heads;
  const int NQ = G * a.q_len;

  grid_dependency_wait();
  const int ctx = checked_context(a, s, threadIdx.x == 0 && split == 0 && kvh == 0);
  const int nblk_seq = (ctx + kBlock - 1) / kBlock;
  const int n_splits = (nblk_seq + a.part_blocks - 1) / a.part_blocks;
  if (ctx == 0) {
    if (split == 0) store_zero_rows<T, D>(a, G, s, kvh, THREADS);
    return;
  }
  if (split >= n_splits) return;
  const int blk0 = split * a.part_blocks;
  const int nblk = min(a.part_blocks, nblk_seq - blk0);

  const uint32_t ring = smem_u32(smem);
  if (threadIdx.x == 0) {
    for (int st = 0; st < NS; ++st) {
      mbar_init(smem_u32(&full_bar[st]), 1);
      mbar_init(smem_u32(&empty_bar[st]), NT);
    }
    fence_barrier_init();
  }
  __syncthreads();

  // physical id of block i of the partition (0 for an id outside the pool)
  const int32_t* table = a.block_tables + static_cast<size_t>(s) * a.max_blocks_per_seq + blk0;
  auto block_id = [&](int i, bool& bad) {
    int id = __ldg(table + i);
    bad = id < 0 || id >= a.num_blocks;
    return bad ? 0 : id;
  };
  // which of the partition's (<= 128) blocks have an id outside the pool, one bit each
  uint32_t badw[4];
#pragma unroll
  for (int c = 0; c < 4; ++c) {
    bool bad = false;
    if (32 * c + lane < nblk) (void)block_id(32 * c + lane, bad);
    badw[c] = __ballot_sync(0xffffffffu, bad);
  }

  bool ok = true;
  float m_ref[2] = {-INFINITY, -INFINITY};
  float l_run[2] = {0.f, 0.f};
  float acc[KS][4];
#pragma unroll
  for (int mt = 0; mt < KS; ++mt) acc[mt][0] = acc[mt][1] = acc[mt][2] = acc[mt][3] = 0.f;
  const int g = lane >> 2;
  const int tq = lane & 3;

  if (warp == PRODUCER) {
    // ---- producer ---------------------------------------------------------
    if (lane == 0) {
      const uint64_t policy = l2_policy_evict_first();
      prefetch_tensormap(&kmap);
      prefetch_tensormap(&vmap);
      int issued = 0;
      for (int i = 0; i < nblk; ++i) {
        const int st = i % NS;
        if (i >= NS && !mbar_wait_bounded(smem_u32(&empty_bar[st]), ((i / NS) - 1) & 1)) {
          ok = false;
          break;
        }
        bool bad;
        const int id = block_id(i, bad);
        if (bad) flag_status(a.status, PA_DEV_BAD_BLOCK_ID);
        const uint32_t bar = smem_u32(&full_bar[st]);
        const uint32_t dst = ring + st * STAGE;
        const int y = (id * a.num_kv_heads + kvh) * kBlock;
        mbar_arrive_expect_tx(bar, STAGE);
#pragma unroll
        for (int b = 0; b < NBOX; ++b) {
          tma_load_2d(dst + b * BOX, &kmap, b * 64, y, bar, policy);
          tma_load_2d(dst + TILE + b * BOX, &vmap, b * 64, y, bar, policy);
        }
        issued = i + 1;
      }
      if (!ok) flag_status(a.status, PA_DEV_WAIT_TIMEOUT);
      // every issued copy lands before the CTA may exit (bounded)
      for (int i = issued - 1; i >= 0 && i >= issued - NS; --i)
        mbar_wait_bounded(smem_u32(&full_bar[i % NS]), (i / NS) & 1, 100000000ull);
    }
  } else {
    // ---- consumer: block group bg, 8 query columns n = 8 * t + (0..7) ------------
    const int t = warp % NT;
    const int bg = warp / NT;
    uint32_t qf[KS][2];
    {
      const int n = 8 * t + g;
      const T* qrow = static_cast<const T*>(a.q) + query_row(a, s, kvh, G, n < NQ ? n : 0) * D;
#pragma unroll
      for (int ks = 0; ks < KS; ++ks) {
        if (n < NQ) {
          qf[ks][0] = *reinterpret_cast<const uint32_t*>(qrow + ks * 16 + 2 * tq);
          qf[ks][1] = *reinterpret_cast<const uint32_t*>(qrow + ks * 16 + 8 + 2 * tq);
        } else {
          qf[ks][0] = qf[ks][1] = 0u;
        }
      }
    }
    int lim[2];
#pragma unroll
    for (int e = 0; e < 2; ++e) {
      const int n = 8 * t + 2 * tq + e;
      lim[e] = n < NQ ? ctx - a.q_len + n / G : ctx - 1;
    }
    float mu[2] = {0.f, 0.f};
    const int k_row = (lane & 7) + ((lane >> 3) & 1) * 8;
    const int k_chk = lane >> 4;
    const int v_row = (lane & 7) + (lane >> 4) * 8;
    const int v_chk = (lane >> 3) & 1;

    for (int i = bg; i < nblk; i += BG) {
      const int st = i % NS;
      const bool got = mbar_wait_bounded(smem_u32(&full_bar[st]), (i / NS) & 1);
      if (!__all_sync(0xffffffffu, got)) {
        ok = false;
        break;
      }
      const uint32_t kt = ring + st * STAGE;
      const uint32_t vt = kt + TILE;
      const uint32_t bw = i < 32 ? badw[0] : i < 64 ? badw[1] : i < 96 ? badw[2] : badw[3];
      int nvalid = ctx - (blk0 + i) * kBlock;
      nvalid = nvalid > kBlock ? kBlock : nvalid;
      if ((bw >> (i & 31)) & 1u) nvalid = 0;

      float sa[4] = {0.f, 0.f, 0.f, 0.f};
      float sb[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
      for (int kp = 0; kp < KS / 2; ++kp) {
        uint32_t ae[4], ao[4];
        const int ce = 4 * kp + k_chk, co = ce + 2;
        ldsm_x4(kt + (ce >> 3) * BOX + swz128(k_row, ce & 7), ae[0], ae[1], ae[2], ae[3]);
        ldsm_x4(kt + (co >> 3) * BOX + swz128(k_row, co & 7), ao[0], ao[1], ao[2], ao[3]);
        Mma<T>::run(sa, ae, qf[2 * kp][0], qf[2 * kp][1]);
        Mma<T>::run(sb, ao, qf[2 * kp + 1][0], qf[2 * kp + 1][1]);
      }
      const int kp0 = (blk0 + i) * kBlock + g, kp1 = kp0 + 8;
      const bool in0 = g < nvalid, in1 = g + 8 < nvalid;
      const float x0 = (in0 && kp0 <= lim[0]) ? (sa[0] + sb[0]) * a.scale_log2 : -INFINITY;
      const float x1 = (in0 && kp0 <= lim[1]) ? (sa[1] + sb[1]) * a.scale_log2 : -INFINITY;
      const float x2 = (in1 && kp1 <= lim[0]) ? (sa[2] + sb[2]) * a.scale_log2 : -INFINITY;
      const float x3 = (in1 && kp1 <= lim[1]) ? (sa[3] + sb[3]) * a.scale_log2 : -INFINITY;

      const bool grow = fmaxf(x0, x2) > m_ref[0] + kLazyV || fmaxf(x1, x3) > m_ref[1] + kLazyV;
      if (__any_sync(0xffffffffu, grow)) {
#pragma unroll
        for (int e = 0; e < 2; ++e) {
          const float mb = warp_max_xor(fmaxf(e ? x1 : x0, e ? x3 : x2), 4, 16);
          const float mn = fmaxf(m_ref[e], mb);
          const float nu = mn == -INFINITY ? 0.f : mn;
          const float al = fast_exp2(m_ref[e] - nu);
          l_run[e] *= al;
#pragma unroll
          for (int mt = 0; mt < KS; ++mt) {
            acc[mt][e] *= al;
            acc[mt][e + 2] *= al;
          }
          m_ref[e] = mn;
          mu[e] = nu;
        }
      }
      // the normaliser sums the same T-rounded weights the PV product uses
      const uint32_t pk0 = Mma<T>::pack(fast_exp2(x0 - mu[0]), fast_exp2(x1 - mu[1]));
      const uint32_t pk1 = Mma<T>::pack(fast_exp2(x2 - mu[0]), fast_exp2(x3 - mu[1]));
      const float2 r0 = Mma<T>::unpack(pk0);
      const float2 r1 = Mma<T>::unpack(pk1);
      l_run[0] += r0.x + r1.x;
      l_run[1] += r0.y + r1.y;
      const uint32_t pb0 = movmatrix_trans(pk0);
      const uint32_t pb1 = movmatrix_trans(pk1);

      const bool partial = nvalid < kBlock;
#pragma unroll
      for (int mt = 0; mt < KS; ++mt) {
        const int ch = 2 * mt + v_chk;
        uint32_t vf[4];
        ldsm_x4_trans(vt + (ch >> 3) * BOX + swz128(v_row, ch & 7), vf[0], vf[1], vf[2], vf[3]);
        if (partial) {
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
      // this warp is done with the stage
      __syncwarp();
      if (lane == 0) mbar_arrive(smem_u32(&empty_bar[st]));
    }
    if (!ok && lane == 0) flag_status(a.status, PA_DEV_WAIT_TIMEOUT);
    l_run[0] = warp_sum_xor(l_run[0], 4, 16);
    l_run[1] = warp_sum_xor(l_run[1], 4, 16);
  }

  // ---- every column has one owner: write it for the store / split-K merge -----
  __syncthreads();   // the ring is no longer read: its space holds the merge buffers
  float* red_o = reinterpret_cast<float*>(smem);
  float* red_m = red_o + BG * NC * D;
  float* red_l = red_m + BG * NC;
  if (warp < PRODUCER) {
    const int bg = warp / NT;
    const int n0 = 8 * (warp % NT) + 2 * tq, n1 = n0 + 1;
#pragma unroll
    for (int mt = 0; mt < KS; ++mt) {
      const int d0 = mt * 16 + g;
      if (n0 < NQ) {
        red_o[(bg * NC + n0) * D + d0] = acc[mt][0];
        red_o[(bg * NC + n0) * D + d0 + 8] = acc[mt][2];
      }
      if (n1 < NQ) {
        red_o[(bg * NC + n1) * D + d0] = acc[mt][1];
        red_o[(bg * NC + n1) * D + d0 + 8] = acc[mt][3];
      }
    }
    if (g == 0) {
      if (n0 < NQ) {
        red_m[bg * NC + n0] = m_ref[0];
        red_l[bg * NC + n0] = l_run[0];
      }
      if (n1 < NQ) {
        red_m[bg * NC + n1] = m_ref[1];
        red_l[bg * NC + n1] = l_run[1];
      }
    }
  }
  __syncthreads();
  cta_merge_store<T, BG, D, NC, THREADS>(a, red_o, red_m, red_l, G, s, kvh, split, n_splits);
}

namespace {

template <typename T, int D, int NT>
cudaError_t launch_verify_t(const DecodeArgs& a, const CUtensorMap& kmap, const CUtensorMap& vmap,
                            cudaStream_t stream) {
  // block groups: as many blocks in flight per CTA as the registers allow
  // (4, 3, 2, 1 groups for 1..4 column tiles: 5, 7, 7, 5 warps); rings of
  // 48 KB (4 CTAs per SM) or 64 KB (3 CTAs per SM) of 8 KB stages at D = 128
  constexpr int BG = NT == 1 ? 4 : NT == 2 ? 3 : NT == 3 ? 2 : 1;
  constexpr int STAGE = 2 * (D / 64) * 16 * 128;
  constexpr int RING = (BG * NT + 1) <= 5 ? 49152 : 65536;
  constexpr int NS = RING / STAGE;
  constexpr int MERGE = BG * 8 * NT * D * 4 + 2 * BG * 8 * NT * 4;
  static_assert(MERGE <= NS * STAGE, "merge buffers must fit in the ring");
  const int smem = NS * STAGE + 1024;
  auto kern = verify_tc_kernel<T, D, NT, BG, NS>;
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
  if (e != cudaSuccess) return e;
  dim3 grid(a.max_splits, a.num_kv_heads, a.num_seqs);
  return launch_pdl(kern, grid, dim3((BG * NT + 1) * 32), smem, stream, kmap, vmap, a);
}

template <typename T, int D>
cudaError_t launch_verify_nt(const DecodeArgs& a, const CUtensorMap& kmap, const CUtensorMap& vmap,
                             cudaStream_t stream) {
  const int cols = (a.num_q_heads / a.num_kv_heads) * a.q_len;
  if (cols <= 8) return launch_verify_t<T, D, 1>(a, kmap, vmap, stream);
  if (cols <= 16) return launch_verify_t<T, D, 2>(a, kmap, vmap, stream);
  if (cols <= 24) return launch_verify_t<T, D, 3>(a, kmap, vmap, stream);
  return launch_verify_t<T, D, 4>(a, kmap, vmap, stream);
}

}  // namespace

cudaError_t launch_verify_tc(const DecodeArgs& a, int dtype, const CUtensorMap& kmap, const CUtensorMap& vmap,
                             cudaStream_t stream) {
  if (dtype == PA_BF16) {
    return a.head_dim == 128 ? launch_verify_nt<__nv_bfloat16, 128>(a, kmap, vmap, stream)
                             : launch_verify_nt<__nv_bfloat16, 64>(a, kmap, vmap, stream);
  }
  return a.head_dim == 128 ? launch_verify_nt<__half, 128>(a, kmap, vmap, stream)
                           : launch_verify_nt<__half, 64>(a, kmap, vmap, stream);
}

}  // namespace pa
