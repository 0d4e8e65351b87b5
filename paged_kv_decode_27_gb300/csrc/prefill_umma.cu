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
//  * One CTA per SM works on two consecutive 128-row query tiles of one head
//    (A = rows 256t..256t+127, B = the next 128), which share every K/V tile
//    they both need; a 1-D grid puts the latest (longest) tile pairs first.
//    Ten warps with fixed roles:
//      warps 0-3 / 4-7  softmax for tile A / B: thread r owns query row r.  It
//                 reads its row of S = Q K^T from tensor memory, applies the
//                 causal mask and the online softmax, writes its row of P
//                 (bf16/fp16) back over S and, when its running max grows,
//                 rescales its row of O;
//      warp 8     TMA producer: K tiles and V tiles of 128 keys (8 pool
//                 blocks, read through the block table, whose entries the warp
//                 loads up front) into two 2-stage rings of 128-byte-swizzled
//                 shared memory;
//      warps 9/10 MMA issuers for tile A / B: S = Q K^T (M=128, N=128, K=D; Q
//                 and K from shared memory) and O += P V (M=128, N=D, K=128; P
//                 from tensor memory, V read MN-major straight from its pool
//                 layout).  One issuer per tile, because issuing stalls while
//                 the tensor pipe is busy and must not hold up the other tile.
//    Producer and issuers block in mbarrier.try_wait on the next input they
//    need, leaving the issue slots to the softmax warps.
//    N = 128 keys per S tile: with the A operand in shared memory a narrower
//    MMA costs as much as this one.
//  * Tensor memory (all 512 columns): per tile one S/P buffer of 128 columns
//    and O (D columns).  The two tiles ping-pong: while one tile's softmax
//    runs, the tensor cores work on the other tile's S and PV.
//  * A K stage is released once every S MMA that reads it completes, a V
//    stage once every PV MMA that reads it completes.
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

constexpr int kRows = 128;     // query rows per tile (MMA M)
constexpr int kKeys = 128;     // keys per K/V tile (8 pool blocks)
constexpr int kStages = 2;     // K and V ring depth
constexpr int kBlocksPerTile = kKeys / 16;
constexpr int kThreads = 352;  // 2 x 4 softmax warps + producer warp + one MMA warp per tile
constexpr int kTmemCols = 512;

template <int D>
struct UmmaLayout {
  static constexpr int NBOX = D / 64;                 // 128-byte column boxes per row
  static constexpr int Q_BYTES = kRows * D * 2;       // one Q tile: [NBOX][128 rows][128 B]
  static constexpr int KT_BYTES = kKeys * D * 2;      // one K (or V) tile: [NBOX][128 rows][128 B]
  static constexpr int K_OFF = 2 * Q_BYTES;
  static constexpr int V_OFF = K_OFF + kStages * KT_BYTES;
  static constexpr int SMEM = V_OFF + kStages * KT_BYTES;
  static constexpr int HALF_Q = kRows * 128;          // one 64-column box strip of Q
  static constexpr int HALF_KT = kKeys * 128;         // one 64-column box strip of K or V
  static constexpr uint32_t TMEM_TILE = 256;          // columns per query tile
  static constexpr uint32_t TMEM_S = 0;               // S: kKeys fp32 columns (P packed over its first half)
  static constexpr uint32_t TMEM_O = kKeys;           // O: D fp32 columns
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
  // k_full[2] v_full[2] | k_empty[2 tiles][2] v_empty[2 tiles][2] | s_full p_full pv_done mma_final [2 tiles].
  // Every waiter waits on a phase that cannot be overtaken before it has
  // waited: a barrier's next phase always depends on the waiter's progress.
  __shared__ __align__(8) uint64_t bars[20];
  __shared__ uint32_t tmem_base_sh;
  __shared__ volatile int abort_sh;
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                             ~static_cast<uintptr_t>(1023));
  const uint32_t sQ = smem_u32(smem);
  const uint32_t sK = sQ + L::K_OFF;
  const uint32_t sV = sQ + L::V_OFF;

  // latest tile pairs first: the pair index descends slowest over the 1-D grid
  const int per_layer = a.num_q_heads * a.num_seqs;
  const int pt = (gridDim.x / per_layer) - 1 - static_cast<int>(blockIdx.x) / per_layer;
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
    if (threadIdx.x == 0 && pt == 0 && hq == 0) flag_status(a.status, PA_DEV_BAD_CONTEXT);
    c = c > cap ? cap : c;
    if (c < n || n > a.max_q_len) return;
  }
  // tile g of the pair: query rows qr0[g] .. qr0[g]+127; n_kt[g] key tiles (0 = no rows)
  int nkt_g[2];
#pragma unroll
  for (int g = 0; g < 2; ++g) {
    const int qr = (2 * pt + g) * kRows;
    nkt_g[g] = qr < n ? (c - n + qr + min(kRows, n - qr) - 1) / kKeys + 1 : 0;
  }
  if (nkt_g[0] == 0) return;
  const int n_kt = nkt_g[1] > nkt_g[0] ? nkt_g[1] : nkt_g[0];

  const uint32_t bar0 = smem_u32(&bars[0]);
  auto k_full = [&](int i) { return bar0 + 8u * i; };
  auto v_full = [&](int i) { return bar0 + 16u + 8u * i; };
  auto k_empty = [&](int g, int i) { return bar0 + 32u + 16u * g + 8u * i; };
  auto v_empty = [&](int g, int i) { return bar0 + 64u + 16u * g + 8u * i; };
  auto s_full = [&](int g) { return bar0 + 96u + 8u * g; };
  auto p_full = [&](int g) { return bar0 + 112u + 8u * g; };
  auto pv_done = [&](int g) { return bar0 + 128u + 8u * g; };
  auto mma_final = [&](int g) { return bar0 + 144u + 8u * g; };

  if (threadIdx.x == 0) {
    for (int i = 0; i < kStages; ++i) {
      mbar_init(k_full(i), 1);
      mbar_init(v_full(i), 1);
    }
    for (int g = 0; g < 2; ++g) {
      for (int i = 0; i < kStages; ++i) {
        mbar_init(k_empty(g, i), 1);
        mbar_init(v_empty(g, i), 1);
      }
      mbar_init(s_full(g), 1);
      mbar_init(p_full(g), 4);
      mbar_init(pv_done(g), 1);
      mbar_init(mma_final(g), 1);
    }
    fence_barrier_init();
    abort_sh = 0;
  }
  // The barriers are ready: the producer starts streaming K/V tiles at once, while
  // the other warps allocate tensor memory and stage Q (they meet on named barrier 1).
  __syncthreads();
  uint32_t tmem = 0;
  if (warp != 8) {
    if (warp == 0) {
      tmem_alloc(smem_u32(&tmem_base_sh), kTmemCols);
      tmem_relinquish();
    }
    // Q tiles -> shared memory in the 128-byte-swizzled K-major layout; every load of a
    // row is in flight before the first store
    if (warp < 8) {
      const int g = warp >> 2;
      const int r = threadIdx.x & 127;
      const int lr = (2 * pt + g) * kRows + r;
      const uint4* src = reinterpret_cast<const uint4*>(static_cast<const T*>(a.q) +
                                                        ((static_cast<size_t>(q0) + lr) * a.num_q_heads + hq) * D);
      const uint32_t qbase = sQ + g * L::Q_BYTES;
      uint4 v[D / 8];
#pragma unroll
      for (int cc = 0; cc < D / 8; ++cc) v[cc] = lr < n ? src[cc] : make_uint4(0u, 0u, 0u, 0u);
#pragma unroll
      for (int cc = 0; cc < D / 8; ++cc) {
        const uint32_t dst = qbase + (cc >> 3) * L::HALF_Q + r * 128 + (((cc & 7) ^ (r & 7)) << 4);
        asm volatile("st.shared.v4.b32 [%0], {%1,%2,%3,%4};" ::"r"(dst), "r"(v[cc].x), "r"(v[cc].y), "r"(v[cc].z),
                     "r"(v[cc].w)
                     : "memory");
      }
      fence_proxy_async_smem();
    }
    tc_fence_before_sync();
    asm volatile("bar.sync 1, %0;" ::"r"(kThreads - 32) : "memory");   // every warp but the producer
    tc_fence_after_sync();
    tmem = tmem_base_sh;
  }

  if (warp == 8) {
    // ------------------------------------------------------------ TMA producer
    // The whole warp runs the loop (lane 0 issues the copies).  Pool row
    // coordinates of the blocks are read up front, 128 blocks at a time, spread
    // over the lanes (lane l holds blocks l, l+32, l+64, l+96 of the chunk).
    if (lane == 0) {
      prefetch_tensormap(&kmap);
      prefetch_tensormap(&vmap);
    }
    const uint64_t policy = l2_policy_evict_last();   // other heads of the group re-read these tiles
    const int oob_row = a.num_blocks * a.num_kv_heads * kBlock;   // rows past the pool read as zero
    const int nblk = n_kt * kBlocksPerTile;
    int yr[4];
    int chunk = -1;
    auto load_chunk = [&](int ch) {
#pragma unroll
      for (int k = 0; k < 4; ++k) {
        const int lb = ch * 128 + k * 32 + lane;
        int y = oob_row;
        if (lb < nblk && lb * kBlock < c) {
          const int id = __ldg(a.block_tables + static_cast<size_t>(s) * a.max_blocks_per_seq + lb);
          if (id >= 0 && id < a.num_blocks)
            y = (id * a.num_kv_heads + kvh) * kBlock;
          else
            flag_status(a.status, PA_DEV_BAD_BLOCK_ID);
        }
        yr[k] = y;
      }
      chunk = ch;
    };
    // One box (16 rows x 128 bytes) per lane: a single issuing thread would
    // serialise the tile's kBlocksPerTile * NBOX tensor copies.
    auto load_tile = [&](const CUtensorMap* map, uint32_t dst, uint32_t bar, int j) {
      const int lb0 = j * kBlocksPerTile;              // a tile's blocks never straddle a 32-block group
      if ((lb0 >> 7) != chunk) load_chunk(lb0 >> 7);
      const int k = (lb0 >> 5) & 3;
      const int v = k == 0 ? yr[0] : k == 1 ? yr[1] : k == 2 ? yr[2] : yr[3];
      const int b = lane % kBlocksPerTile;
      const int h = lane / kBlocksPerTile;
      const int y = __shfl_sync(0xffffffffu, v, (lb0 + b) & 31);
      if (lane == 0) mbar_arrive_expect_tx(bar, L::KT_BYTES);
      __syncwarp();
      if (h < NBOX) tma_load_2d(dst + h * L::HALF_KT + b * 2048, map, h * 64, y, bar, policy);
      __syncwarp();
    };
    // Fixed order K_0 V_0 K_1 V_1 ...: K_{j+2} reuses the stage freed by the S
    // MMAs of tile j, V_{j+2} the one freed by its PV MMAs.  The warp blocks
    // (suspended in mbarrier.try_wait) on exactly the next release it needs.
    auto stage_free = [&](bool is_k, int j) -> bool {   // all lanes
      if (j < kStages) return true;
      const int jp = j - kStages;
      bool ok2 = true;
#pragma unroll
      for (int g = 0; g < 2; ++g)
        if (jp < nkt_g[g])
          ok2 = ok2 && !abort_sh &&
                mbar_wait_bounded(is_k ? k_empty(g, jp % kStages) : v_empty(g, jp % kStages), (jp / kStages) & 1);
      return __all_sync(0xffffffffu, ok2) != 0;
    };
    int next_k = 0, next_v = 0;
    load_chunk(0);
    for (int j = 0; j < n_kt; ++j) {
      if (!stage_free(true, j)) {
        abort_sh = 1;
        break;
      }
      load_tile(&kmap, sK + (j % kStages) * L::KT_BYTES, k_full(j % kStages), j);
      next_k = j + 1;
      if (!stage_free(false, j)) {
        abort_sh = 1;
        break;
      }
      load_tile(&vmap, sV + (j % kStages) * L::KT_BYTES, v_full(j % kStages), j);
      next_v = j + 1;
    }
    if (abort_sh && lane == 0) {
      // let the copies still in flight land before the CTA can exit
      for (int j = next_k - kStages < 0 ? 0 : next_k - kStages; j < next_k; ++j)
        mbar_wait_bounded(k_full(j % kStages), (j / kStages) & 1, 100000000ull);
      for (int j = next_v - kStages < 0 ? 0 : next_v - kStages; j < next_v; ++j)
        mbar_wait_bounded(v_full(j % kStages), (j / kStages) & 1, 100000000ull);
    }
  } else if (warp >= 9) {
    // ----------------------------------------------------- MMA issuer, one per tile
    const int g = warp - 9;
    const uint32_t tt = tmem + g * L::TMEM_TILE;
    const uint32_t id_s = umma_idesc_f16(kRows, kKeys, kBf16, false, false);
    const uint32_t id_o = umma_idesc_f16(kRows, D, kBf16, false, true);
    // With one S/P buffer per tile the order is fixed -- S_0, PV_0, S_1, PV_1,
    // ... -- so the warp blocks (suspended in mbarrier.try_wait, taking no
    // issue slots from the softmax warps) on exactly the next input it needs.
    bool ok = true;
    const int my_nkt = nkt_g[g];
    auto wait_all = [&](uint32_t bar, uint32_t parity) -> bool {
      return __all_sync(0xffffffffu, !abort_sh && mbar_wait_bounded(bar, parity)) != 0;
    };
    for (int j = 0; j < my_nkt && ok; ++j) {
      const int st = j % kStages;
      // S_j = Q K_j^T once K_j has landed and PV_{j-1} (which read P from the
      // same columns) has completed
      ok = wait_all(k_full(st), (j / kStages) & 1) && (j < 1 || wait_all(pv_done(g), (j - 1) & 1));
      // Tile B starts once tile A's first softmax is done, so that the two tiles run out of
      // phase (one tile's MMAs during the other's softmax) instead of in step on every K tile.
      if (ok && g == 1 && j == 0) ok = wait_all(p_full(0), 0);
      if (!ok) break;
      tc_fence_after_sync();
      if (lane == 0) {
        const uint32_t qbase = sQ + g * L::Q_BYTES;
        const uint32_t kbase = sK + st * L::KT_BYTES;
#pragma unroll
        for (int kk = 0; kk < D / 16; ++kk) {
          const uint64_t da = umma_desc_sw128(qbase + (kk >> 2) * L::HALF_Q + (kk & 3) * 32, 16, 1024);
          const uint64_t db = umma_desc_sw128(kbase + (kk >> 2) * L::HALF_KT + (kk & 3) * 32, 16, 1024);
          umma_f16(tt + L::TMEM_S, da, db, id_s, kk > 0 ? 1u : 0u);
        }
        umma_commit(s_full(g));
        umma_commit(k_empty(g, st));
      }
      __syncwarp();
      // O += P_j V_j once V_j has landed and the softmax has written P_j
      ok = wait_all(v_full(st), (j / kStages) & 1) && wait_all(p_full(g), j & 1);
      if (!ok) break;
      const uint32_t vbase = sV + st * L::KT_BYTES;
      const int pb = c >> 4;
      if ((c & 15) && pb / kBlocksPerTile == j) {
        // value rows past the context read as zero (both issuers write the
        // same zeros; each does it before its own PV reads the tile)
        const int r0 = c & 15;
        for (int idx = lane; idx < (16 - r0) * NBOX * 8; idx += 32) {
          const int row = (pb % kBlocksPerTile) * 16 + r0 + idx / (NBOX * 8);
          const int rem = idx % (NBOX * 8);
          const uint32_t addr = vbase + (rem >> 3) * L::HALF_KT + row * 128 + ((rem & 7) << 4);
          asm volatile("st.shared.v4.b32 [%0], {%1,%1,%1,%1};" ::"r"(addr), "r"(0u) : "memory");
        }
        fence_proxy_async_smem();
      }
      __syncwarp();
      tc_fence_after_sync();
      if (lane == 0) {
        const uint32_t ptm = tt + L::TMEM_S;   // P: kKeys/2 columns of packed pairs
#pragma unroll
        for (int kk = 0; kk < kKeys / 16; ++kk) {
          const uint64_t db = umma_desc_sw128(vbase + kk * 2048, L::HALF_KT, 1024);
          umma_f16_tmem_a(tt + L::TMEM_O, ptm + kk * 8, db, id_o, (j > 0 || kk > 0) ? 1u : 0u);
        }
        umma_commit(pv_done(g));
        umma_commit(v_empty(g, st));
      }
      __syncwarp();
    }
    if (!ok) abort_sh = 1;
    // every MMA issued by this warp has completed before the CTA tears down
    if (lane == 0) umma_commit(mma_final(g));
    mbar_wait_bounded(mma_final(g), 0, 100000000ull);
  } else {
    // ----------------------------------------------------------- softmax warps
    const int g = warp >> 2;
    const int r = threadIdx.x & 127;
    const int qr0 = (2 * pt + g) * kRows;
    const int lr = qr0 + r;
    const int pos = c - n + lr;                       // causal limit of this row
    const int my_nkt = nkt_g[g];
    const uint32_t tt = tmem + g * L::TMEM_TILE;
    const uint32_t lane_base = static_cast<uint32_t>((warp & 3) * 32) << 16;
    const uint32_t tO = tt + L::TMEM_O + lane_base;
    float m_used = -INFINITY;   // reference max of this row (log2 domain)
    float l = 0.f;              // sum of 2^(x - m_used)
    bool ok = true;
    // scale > 0 (the usual case): the max is taken on the raw scores and the
    // scale folds into one FMA per element; otherwise scale first.
    const bool pos_scale = a.scale_log2 > 0.f;
    const int warp_pos_min = c - n + qr0 + (warp & 3) * 32;   // smallest causal limit in this warp
    const uint32_t tbuf = tt + L::TMEM_S + lane_base;
    const float sc = pos_scale ? a.scale_log2 : 1.f;   // p = 2^(x*sc - mu) on raw scores x
    for (int j = 0; j < my_nkt; ++j) {
      ok = !abort_sh && mbar_wait_bounded(s_full(g), j & 1);
      if (!__all_sync(0xffffffffu, ok)) {
        ok = false;
        break;
      }
      tc_fence_after_sync();
      const int key0 = j * kKeys;
      const bool diag = key0 + kKeys - 1 > warp_pos_min;   // a tile on the diagonal: causal mask
      // the whole row of S in one tensor-memory load
      float x[kKeys];
      tmem_ld128(tbuf, x);
      if (!pos_scale) {
#pragma unroll
        for (int i = 0; i < kKeys; ++i) x[i] *= a.scale_log2;
      }
      if (diag) {
#pragma unroll
        for (int i = 0; i < kKeys; ++i)
          if (key0 + i > pos) x[i] = -INFINITY;
      }
      float pm[8];
#pragma unroll
      for (int k = 0; k < 8; ++k) pm[k] = x[k];
#pragma unroll
      for (int i = 8; i < kKeys; i += 8)
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
        // rescale this warp's rows of O; PV_{j-1} has completed (S_j waited for it)
        ok = mbar_wait_bounded(pv_done(g), (j - 1) & 1);
        if (!__all_sync(0xffffffffu, ok)) {
          ok = false;
          break;
        }
        tc_fence_after_sync();
#pragma unroll 1
        for (int cc = 0; cc < D / 16; ++cc) {   // 16 columns at a time: the row of S is still live
          float o[16];
          tmem_ld16(tO + cc * 16, o);
          uint32_t ob[16];
#pragma unroll
          for (int i = 0; i < 16; ++i) ob[i] = __float_as_uint(o[i] * factor);
          tmem_st16_u(tO + cc * 16, ob);
        }
      }
      const float mu = (m_used == -INFINITY) ? 0.f : m_used;
      // P = 2^(x - mu), packed two per column over the front of S
      float ps[8] = {0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f};   // independent partial sums
#pragma unroll
      for (int cc = 0; cc < kKeys / 32; ++cc) {
        uint32_t w[16];
#pragma unroll
        for (int i = 0; i < 16; ++i) {
          const float p0 = fast_exp2(fmaf(x[cc * 32 + 2 * i], sc, -mu));
          const float p1 = fast_exp2(fmaf(x[cc * 32 + 2 * i + 1], sc, -mu));
          ps[(2 * i) & 7] += p0;
          ps[(2 * i + 1) & 7] += p1;
          w[i] = Mma<T>::pack(p0, p1);
        }
        tmem_st16_u(tbuf + cc * 16, w);   // keys 32cc+2i, 32cc+2i+1 in column 16cc+i
      }
      l += ((ps[0] + ps[1]) + (ps[2] + ps[3])) + ((ps[4] + ps[5]) + (ps[6] + ps[7]));
      tmem_wait_st();
      tc_fence_before_sync();
      __syncwarp();
      if (lane == 0) mbar_arrive(p_full(g));
    }
    if (!ok) {
      abort_sh = 1;
    } else if (my_nkt > 0) {
      // the last PV (and so every PV before it) has completed
      ok = mbar_wait_bounded(pv_done(g), (my_nkt - 1) & 1);
      if (__all_sync(0xffffffffu, ok)) {
        tc_fence_after_sync();
        const float inv = l > 0.f ? 1.f / l : 0.f;
        T* orow = static_cast<T*>(a.out) + ((static_cast<size_t>(q0) + lr) * a.num_q_heads + hq) * D;
#pragma unroll
        for (int cc = 0; cc < D / 32; ++cc) {
          float o[32];
          tmem_ld32(tO + cc * 32, o);
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
  const long long n_pairs = ((a.max_q_len + kRows - 1) / kRows + 1) / 2;
  const long long ctas = n_pairs * a.num_q_heads * a.num_seqs;
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
