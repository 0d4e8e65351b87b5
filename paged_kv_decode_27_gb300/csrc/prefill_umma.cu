// prefill_umma.cu -- causal prompt attention over the paged pool on the 5th-
// generation tensor cores (tcgen05, accumulators in tensor memory).
//
// The prompt pass processes all prompt tokens at once (q_len = prompt length,
// "LLM Inference Server", Stage 1) under a causal mask ("LLM Inference Server
// From Scratch", What you build: fused attention with causal masking; How it
// works, 4 Attention Kernel: causal mask, GQA).  It is a dense contraction and
// compute-bound ("LLM Inference Server", What You Will Build), so it runs on
// tcgen05.mma.
//
// Work.  One item = one 128-row query tile of one sequence for two q heads of
// the same KV head (tile A = head 2p, tile B = head 2p + 1; one head per item
// when the query group is odd).  The two tiles need the same K/V tiles in the
// same order and as many of them, so every K/V tile is read into shared
// memory once for both: the bytes an SM receives per product are what bound
// this kernel once its MMAs are pipelined.  The grid is persistent (one CTA
// per SM): each CTA sorts the (sequence, query tile) pairs by their number of
// key tiles, longest first, in shared memory, and the items (a pair and a
// head pair) are handed out at run time in that order from a global counter,
// each to the first CTA with room for it.
//
// Per K tile j of an item (128 keys = 8 pool blocks) and per tile g:
//   S_g = Q_g K^T  (M = 128 query rows, N = 128 keys, K = D; Q and K from
//                   128-byte swizzled shared memory) into tensor memory;
//   softmax        one thread per query row reads its row of S, applies the
//                   causal mask (a select per key on the diagonal tile: the
//                   rows of a warp differ, a branch would diverge) and the
//                   online softmax (log2 domain, the running reference raised
//                   lazily: only when a row's maximum grows by more than
//                   2^8), writes P (bf16/fp16 pairs) over S;
//   O_g += P_g V   (M = 128, N = D, K = 128 keys; P from tensor memory, V read
//                   MN-major straight from its pool layout).
// One thread issues both tiles' products, interleaved so that one tile's
// products run during the other's softmax.  It issues S for K tile j + 1
// right after PV for tile j: the MMAs of one thread run in issue order, so
// S_{j+1} overwrites the columns of P_j only after PV_j has read them, and
// the next S needs no wait on the PV's completion.  The same order makes the
// completion of S_g(j) imply that of every product issued before it (PV of
// both tiles for K tile j - 1), so the softmax needs no separate signal for
// the previous PV and hands the K and V stages back to the producers itself.
// The tensor core accepts barely more than one MMA ahead of the one it runs,
// so every wait or branch of the issuing thread between two products leaves
// the pipe idle: the issuer is one thread with precomputed descriptors and
// two commits per K tile (S of each tile).
//
// Tensor memory (512 columns): per tile S/P (128 columns) and O (D columns).
// Shared memory: Q_A, Q_B, a 2-stage K ring and a 3-stage V ring, the sorted
// work list (its histogram space then holds the ring of published items).
//
// Warps (384 threads, three warpgroups that re-balance their registers with
// setmaxnreg):
//   0-3 / 4-7  softmax of tile A / B (thread r owns query row r), and at the
//              end of an item the epilogue: normalise O and store the rows
//              (32-byte stores when the output is 32-byte aligned); the next
//              item is taken from the ring while the item's last PV runs
//              (for bf16 queries over an fp16 pool, also the in-place
//              conversion of the tile's next Q, done while the item's last
//              PV runs, so that the next item's S overlaps the epilogue);
//   8 / 10     TMA producers of the K ring / the V ring (pool rows through the
//              block table);
//   9          MMA issuer of both tiles (lane 0 alone), in the interleaved
//              order below;
//   11         query loader and scheduler: takes the items (the first by
//              CTA index, the rest from the global counter), publishes them
//              decoded into the ring, and loads each item's Q tiles (TMA;
//              cp.async for a prompt's last partial tile) once the previous
//              item's S products have completed.
// Every hand-off is an mbarrier; every wait is bounded, and a timeout sets
// PA_DEV_WAIT_TIMEOUT, lets the copies and MMAs in flight finish (bounded)
// and frees the tensor memory.
//
// Query i of a sequence with context c and q_len n sits at position
// c - n + i and sees keys 0..c - n + i; value rows past the context are zeroed
// in shared memory (and whole blocks past it read as zero), so stale pool data
// never reaches the output.
#include <type_traits>

#include "pa_common.cuh"
#include "pa_internal.h"

namespace pa {

namespace {

constexpr int kRows = 128;      // query rows per tile (MMA M)
constexpr int kKeys = 128;      // keys per K/V tile (MMA N of S, K of PV)
constexpr int kStagesK = 2;     // K ring depth
constexpr int kStagesV = 3;     // V ring depth: a V stage waits longest to be refilled (the PV of both tiles)
constexpr int kBlocksPerTile = kKeys / 16;
constexpr int kThreads = 384;   // three warpgroups
constexpr int kTmemCols = 512;
constexpr int kMaxPairs = 384;    // (sequence, query tile) pairs sorted in shared memory
constexpr int kMaxCost = 63;      // key tiles per query tile, for the sort's buckets (longer share the last)
constexpr int kRing = 4;          // item indices published ahead by the query loader
constexpr int kRingEntry = 8;     // ints per ring entry: index, then the item's s h t q0 n c nkt
static_assert(kRing * kRingEntry * 4 + 2 * kRing * 8 <= (kMaxCost + 1) * 4, "the item ring fits the sort's histogram");
// Registers per thread after the warpgroups re-balance the launch's
// 168 x 384 = 64512: (200 + 200 + 96) x 128 = 63488 <= 64512, so the
// increases never wait for registers that are not there.
constexpr int kRegsSoftmax = 200;
constexpr int kRegsIo = 96;
static_assert((2 * kRegsSoftmax + kRegsIo) * 128 <= 168 * kThreads, "register split");

template <int D>
struct UmmaLayout {
  static constexpr int NBOX = D / 64;                 // 128-byte column boxes per row
  static constexpr int Q_BYTES = kRows * D * 2;       // one Q tile: [NBOX][128 rows][128 B]
  static constexpr int KT_BYTES = kKeys * D * 2;      // one K (or V) tile: [NBOX][128 rows][128 B]
  static constexpr int HALF_Q = kRows * 128;          // one 64-column box strip of Q
  static constexpr int HALF_KT = kKeys * 128;         // one 64-column box strip of K or V
  static constexpr int K_OFF = 2 * Q_BYTES;
  static constexpr int V_OFF = K_OFF + kStagesK * KT_BYTES;
  static constexpr int PAIRS_OFF = V_OFF + kStagesV * KT_BYTES;  // int32 [kMaxPairs]
  static constexpr int HIST_OFF = PAIRS_OFF + kMaxPairs * 4;     // int32 [kMaxCost + 1]
  static constexpr int SMEM = HIST_OFF + (kMaxCost + 1) * 4;
  static constexpr uint32_t TMEM_TILE = 256;          // columns per query tile
  static constexpr uint32_t TMEM_S = 0;               // S: kKeys fp32 columns (P packed over its first half)
  static constexpr uint32_t TMEM_O = kKeys;           // O: D fp32 columns
};

// One work item: query tile t (rows 128t ..) of sequence s, q heads h (tile A)
// and h + 1 (tile B, when paired).
struct Item {
  int s, h, t, q0, n, c, nkt;
};

__device__ __forceinline__ int key_tiles(int c, int n, int t) {
  // the tile's last row sits at position c - n + min(128 (t + 1), n) - 1
  return (c - n + min(kRows * (t + 1), n) - 1) / kKeys + 1;
}

}  // namespace

// T: the type of the pool and of the products' operands; TA: the type of q
// and of the output rows (T, or bf16 for an fp16 pass over bf16 activations:
// the query loader then converts each Q tile in shared memory).
template <typename T, typename TA, int D>
__global__ void __launch_bounds__(kThreads, 1)
prefill_umma_kernel(const __grid_constant__ CUtensorMap kmap, const __grid_constant__ CUtensorMap vmap,
                    const __grid_constant__ CUtensorMap qmap, const PrefillArgs a) {
  using L = UmmaLayout<D>;
  constexpr int NBOX = L::NBOX;
  constexpr bool kBf16 = !std::is_same<T, __half>::value;
  constexpr bool kCvtQ = !std::is_same<T, TA>::value;   // bf16 queries into an fp16 pass

  extern __shared__ uint8_t smem_raw[];
  // k_full[2] k_empty[2] v_full[3] v_empty[3] | s_full[2] p_full[2] pv_done[2] o_free[2] |
  // q_full[2] q_empty[2] | mma_final | q_raw[2]
  __shared__ __align__(8) uint64_t bars[kCvtQ ? 25 : 23];
  __shared__ uint32_t tmem_base_sh;
  __shared__ volatile int abort_sh;
  __shared__ int n_pairs_sh;
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                             ~static_cast<uintptr_t>(1023));
  const uint32_t sQ = smem_u32(smem);
  const uint32_t sK = sQ + L::K_OFF;
  const uint32_t sV = sQ + L::V_OFF;
  int* pairs = reinterpret_cast<int*>(smem + L::PAIRS_OFF);
  int* hist = reinterpret_cast<int*>(smem + L::HIST_OFF);

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const int H = a.num_q_heads;
  const int G = H / a.num_kv_heads;
  const bool paired = (G % 2) == 0;     // tile B exists
  const int NT = paired ? 2 : 1;        // query tiles per item
  const int HG = H / NT;                // head groups per (sequence, query tile)

  const uint32_t bar0 = smem_u32(&bars[0]);
  auto k_full = [&](int i) { return bar0 + 8u * i; };
  auto k_empty = [&](int i) { return bar0 + 16u + 8u * i; };
  auto v_full = [&](int i) { return bar0 + 32u + 8u * i; };
  auto v_empty = [&](int i) { return bar0 + 56u + 8u * i; };
  auto s_full = [&](int g) { return bar0 + 80u + 8u * g; };
  auto p_full = [&](int g) { return bar0 + 96u + 8u * g; };
  auto pv_done = [&](int g) { return bar0 + 112u + 8u * g; };
  auto o_free = [&](int g) { return bar0 + 128u + 8u * g; };
  auto q_full = [&](int g) { return bar0 + 144u + 8u * g; };
  auto q_empty = [&](int g) { return bar0 + 160u + 8u * g; };
  auto mma_final = [&](int g) { return bar0 + 176u + 8u * g; };
  auto q_raw = [&](int g) { return bar0 + 184u + 8u * g; };   // a Q tile landed, before its conversion

  if (threadIdx.x == 0) {
    for (int i = 0; i < kStagesK; ++i) {
      mbar_init(k_full(i), 1);
      mbar_init(k_empty(i), 1);   // released by the last tile's softmax once the S products of the tile have completed
    }
    for (int i = 0; i < kStagesV; ++i) {
      mbar_init(v_full(i), 1);
      mbar_init(v_empty(i), 1);
    }
    for (int g = 0; g < 2; ++g) {
      mbar_init(s_full(g), 1);
      mbar_init(p_full(g), 4);
      mbar_init(pv_done(g), 1);
      mbar_init(o_free(g), 4);
      mbar_init(q_full(g), kCvtQ ? 4 : 1);   // the TMA, or the tile's four softmax warps after the conversion
      mbar_init(q_empty(g), 1);
      if (kCvtQ) mbar_init(q_raw(g), 1);
    }
    mbar_init(mma_final(0), 1);
    fence_barrier_init();
    abort_sh = 0;
    n_pairs_sh = 0;
  }
  if (warp == 0) {
    __syncwarp();   // thread 0 has left the set-up above: the allocation is warp-wide
    tmem_alloc(smem_u32(&tmem_base_sh), kTmemCols);
    tmem_relinquish();
  }
  if (warp == 8 && lane == 0) prefetch_tensormap(&kmap);
  if (warp == 10 && lane == 0) prefetch_tensormap(&vmap);
  if (warp == 11 && lane == 0) prefetch_tensormap(&qmap);

  grid_dependency_wait();   // the prompt's K/V were appended by the kernel before us

  // ---- the work list: (sequence, query tile) pairs sorted by key tiles, most
  // first (a counting sort; within a bucket the order does not matter).
  const int cap = a.max_blocks_per_seq * kBlock;
  auto seq_load = [&](int s, int& q0, int& n, int& c) {
    q0 = __ldg(a.cu_q_lens + s);
    n = __ldg(a.cu_q_lens + s + 1) - q0;
    c = __ldg(a.context_lens + s);
  };
  auto seq_shape = [&](int s, int& q0, int& n, int& c) -> bool {
    seq_load(s, q0, n, c);
    return n > 0 && n <= a.max_q_len && c >= n && c <= cap;
  };
  for (int i = threadIdx.x; i <= kMaxCost; i += kThreads) hist[i] = 0;
  __syncthreads();
  for (int s = threadIdx.x; s < a.num_seqs; s += kThreads) {
    int q0, n, c;
    const bool ok = seq_shape(s, q0, n, c);
    if (!ok && !(n == 0 && c >= 0 && c <= cap) && blockIdx.x == 0) flag_status(a.status, PA_DEV_BAD_CONTEXT);
    if (!ok) continue;
    const int nt = (n + kRows - 1) / kRows;
    atomicAdd(&n_pairs_sh, nt);
    for (int t = 0; t < nt; ++t) atomicAdd(&hist[min(key_tiles(c, n, t), kMaxCost)], 1);
  }
  __syncthreads();
  const int n_pairs = n_pairs_sh;
  const bool sorted = n_pairs <= kMaxPairs;
  if (sorted) {
    if (warp == 0) {
      // exclusive prefix over the buckets, most key tiles first: lane l sums a
      // contiguous run of 32 buckets (from the top), then a warp scan
      const int per = (kMaxCost + 1) / 32;
      const int hi = kMaxCost - lane * per;   // this lane's buckets: hi, hi-1, ..., hi-per+1
      int run = 0;
      for (int i = 0; i < per; ++i) run += hist[hi - i];
      int incl = run;
#pragma unroll
      for (int o = 1; o < 32; o <<= 1) {
        const int v = __shfl_up_sync(0xffffffffu, incl, o);
        if (lane >= o) incl += v;
      }
      int off = incl - run;
      for (int i = 0; i < per; ++i) {
        const int cnt = hist[hi - i];
        hist[hi - i] = off;
        off += cnt;
      }
    }
    __syncthreads();
    for (int s = threadIdx.x; s < a.num_seqs; s += kThreads) {
      int q0, n, c;
      if (!seq_shape(s, q0, n, c)) continue;
      const int nt = (n + kRows - 1) / kRows;
      for (int t = 0; t < nt; ++t) {
        const int pos = atomicAdd(&hist[min(key_tiles(c, n, t), kMaxCost)], 1);
        pairs[pos] = (s << 16) | t;
      }
    }
  }
  // Without the sorted list (too many pairs), items run over every
  // (query tile, sequence, head group) in order of decreasing tile, skipping empty ones.
  const int t_max = (a.max_q_len + kRows - 1) / kRows;
  const long long n_items = sorted ? static_cast<long long>(n_pairs) * HG
                                   : static_cast<long long>(t_max) * a.num_seqs * HG;
  // Items are handed out at run time, longest first: CTA b starts with item
  // b, and then the query loader of a CTA takes the next item index from a
  // global counter when its CTA has room for another, so a CTA that drew
  // short items takes more of them (a longest-processing-time schedule,
  // without knowing the items' times).  The loader publishes each item (its
  // index and decoded fields) into a 4-entry ring in shared memory (kRing),
  // read by the other roles in the same order, so no reader decodes an item
  // from global memory; index -1 ends the ring.
  // item_at: item k of the list; false when it has no work.
  auto item_at = [&](int k, Item& it) -> bool {
    it.h = (k % HG) * NT;
    if (sorted) {
      const int p = pairs[k / HG];
      it.s = p >> 16;
      it.t = p & 0xffff;
    } else {
      const int r = k / HG;
      it.s = r % a.num_seqs;
      it.t = t_max - 1 - r / a.num_seqs;
    }
    if (!seq_shape(it.s, it.q0, it.n, it.c)) return false;
    if (it.t * kRows >= it.n) return false;
    it.nkt = key_tiles(it.c, it.n, it.t);
    return true;
  };
  // The ring lives where the sort's histogram was (free from here on).
  int* ring = hist;
  const uint32_t ring_bar = smem_u32(hist + kRing * kRingEntry);   // item_full[kRing] item_empty[kRing]
  auto item_full = [&](int i) { return ring_bar + 8u * i; };
  auto item_empty = [&](int i) { return ring_bar + 8u * (kRing + i); };
  // A reader's read number `use`: every reading thread waits for the entry
  // (bounded) and copies it; one thread per reading warp hands the slot back
  // once the warp has read it.  ring_get returns the index (-1: the end).
  auto ring_wait = [&](uint32_t use) -> bool {
    return !abort_sh && mbar_wait_bounded(item_full(static_cast<int>(use % kRing)), (use / kRing) & 1);
  };
  auto ring_get = [&](uint32_t use, Item& x) -> int {
    const volatile int* e = ring + kRingEntry * static_cast<int>(use % kRing);
    x.s = e[1];
    x.h = e[2];
    x.t = e[3];
    x.q0 = e[4];
    x.n = e[5];
    x.c = e[6];
    x.nkt = e[7];
    return e[0];
  };
  auto ring_release = [&](uint32_t use) { mbar_arrive(item_empty(static_cast<int>(use % kRing))); };

  tc_fence_before_sync();
  __syncthreads();
  tc_fence_after_sync();
  const uint32_t tmem = tmem_base_sh;
  // every thread is done with the histogram: the ring's barriers take its place
  if (threadIdx.x == 0) {
    for (int i = 0; i < kRing; ++i) {
      mbar_init(item_full(i), 1);
      mbar_init(item_empty(i), 3 + 4 * NT);   // K and V producers, issuer, every softmax warp
    }
    fence_barrier_init();
  }
  __syncthreads();

  // Each role branch starts by setting its warpgroup's registers (every warp
  // of a warpgroup takes the same setmaxnreg) and ends with the CTA-wide
  // teardown barrier (named barrier 1, all threads).
  auto teardown = [&]() {
    __syncwarp();
    tc_fence_before_sync();
    asm volatile("bar.sync 1, %0;" ::"n"(kThreads) : "memory");
  };

  if (warp >= 8) {
    asm volatile("setmaxnreg.dec.sync.aligned.u32 %0;" ::"n"(kRegsIo));
    if (warp == 8 || warp == 10) {
      // --------------------------------------------- TMA producers: K (8), V (10)
      // Each ring has its own producer, so a K tile waits only for the S
      // products of the tile two before it and a V tile only for the PV
      // products (the last tile's softmax releases both, see the issuer).  The whole warp runs the loop (one box per lane).  Pool row
      // coordinates of an item's blocks are read 128 blocks at a time, spread
      // over the lanes (lane l holds blocks l, l+32, l+64, l+96 of the chunk).
      const bool is_k = warp == 8;
      const CUtensorMap* map = is_k ? &kmap : &vmap;
      const uint32_t ring_base = is_k ? sK : sV;
      const uint32_t nst = is_k ? kStagesK : kStagesV;
      const uint64_t policy = l2_policy_evict_last();   // the other heads of the group read these tiles too
      const int oob_row = a.num_blocks * a.num_kv_heads * kBlock;   // rows past the pool read as zero
      uint32_t kv = 0;       // tiles issued
      bool ok = true;
      uint32_t use = 0;      // ring reads
      Item it;
      auto wait_all = [&](uint32_t bar, uint32_t parity) -> bool {
        return __all_sync(0xffffffffu, !abort_sh && mbar_wait_bounded(bar, parity)) != 0;
      };
      // the next item from the ring, read by the whole warp
      auto next = [&]() -> int {
        if (!__all_sync(0xffffffffu, ring_wait(use))) return -2;
        const int kk = ring_get(use, it);
        __syncwarp();
        if (lane == 0) ring_release(use);
        ++use;
        return kk;
      };
      int kc;
      while (ok && (kc = next()) >= 0) {
        const int kvh = it.h / G;
        const int nblk = it.nkt * kBlocksPerTile;
        int yr[4];
        int chunk = -1;
        auto load_chunk = [&](int ch) {
#pragma unroll
          for (int q = 0; q < 4; ++q) {
            const int lb = ch * 128 + q * 32 + lane;
            int y = oob_row;
            if (lb < nblk && lb * kBlock < it.c) {
              const int id = __ldg(a.block_tables + static_cast<size_t>(it.s) * a.max_blocks_per_seq + lb);
              if (id >= 0 && id < a.num_blocks)
                y = (id * a.num_kv_heads + kvh) * kBlock;
              else
                flag_status(a.status, PA_DEV_BAD_BLOCK_ID);
            }
            yr[q] = y;
          }
          chunk = ch;
        };
        // One box (16 rows x 128 bytes) per lane: a single issuing thread
        // would serialise the tile's kBlocksPerTile * NBOX tensor copies.
        auto load_tile = [&](const CUtensorMap* map, uint32_t dst, uint32_t bar, int j) {
          const int lb0 = j * kBlocksPerTile;   // a tile's blocks never straddle a 32-block group
          if ((lb0 >> 7) != chunk) load_chunk(lb0 >> 7);
          const int q = (lb0 >> 5) & 3;
          const int v = q == 0 ? yr[0] : q == 1 ? yr[1] : q == 2 ? yr[2] : yr[3];
          const int b = lane % kBlocksPerTile;
          const int h = lane / kBlocksPerTile;
          const int y = __shfl_sync(0xffffffffu, v, (lb0 + b) & 31);
          if (lane == 0) mbar_arrive_expect_tx(bar, L::KT_BYTES);
          __syncwarp();
          if (h < NBOX) tma_load_2d(dst + h * L::HALF_KT + b * 2048, map, h * 64, y, bar, policy);
          __syncwarp();
        };
        for (int j = 0; j < it.nkt; ++j) {
          const int st = static_cast<int>(kv % nst);
          const uint32_t use = kv / nst;
          // stage st is free once the products of its previous use have completed
          if (use > 0 && !wait_all(is_k ? k_empty(st) : v_empty(st), (use - 1) & 1)) {
            ok = false;
            break;
          }
          load_tile(map, ring_base + st * L::KT_BYTES, is_k ? k_full(st) : v_full(st), j);
          ++kv;
        }
      }
      if (kc == -2) ok = false;
      if (!ok) {
        abort_sh = 1;
        // let the copies still in flight (at most the last kStages of each
        // ring) land before the CTA can exit
        if (lane == 0)
          for (uint32_t u = kv > nst ? kv - nst : 0; u < kv; ++u)
            mbar_wait_bounded(is_k ? k_full(u % nst) : v_full(u % nst), (u / nst) & 1, 100000000ull);
      }
    } else if (warp == 9) {
      // ------------------------------------------------------------ MMA issuer
      // One thread (lane 0) issues both tiles' products in a fixed interleaved order:
      //   S_A0 S_B0 | PV_A0 S_A1 PV_B0 S_B1 | PV_A1 S_A2 PV_B1 S_B2 | ...
      if (lane == 0) {
        const uint32_t id_s = umma_idesc_f16(kRows, kKeys, kBf16, false, false);
        const uint32_t id_o = umma_idesc_f16(kRows, D, kBf16, false, true);
        // a wait whose phase has already completed costs one try_wait; the abort
        // flag is read only when the wait has to block
        auto wait1 = [&](uint32_t bar, uint32_t parity) -> bool {
          return mbar_try_wait(bar, parity) || (!abort_sh && mbar_wait_bounded(bar, parity));
        };
        // descriptors of the operand bases; the start address field (bits 0-13,
        // 16-byte units) takes the in-tile offsets by plain addition
        const uint64_t dq = umma_desc_sw128(sQ, 16, 1024);
        const uint64_t dk = umma_desc_sw128(sK, 16, 1024);
        const uint64_t dv = umma_desc_sw128(sV, L::HALF_KT, 1024);
        auto issue_s = [&](int g, int st) {
          tc_fence_after_sync();
          const uint64_t ba = dq + static_cast<uint64_t>((g * L::Q_BYTES) >> 4);
          const uint64_t bb = dk + static_cast<uint64_t>((st * L::KT_BYTES) >> 4);
          const uint32_t td = tmem + g * L::TMEM_TILE + L::TMEM_S;
#pragma unroll
          for (int kk = 0; kk < D / 16; ++kk) {
            umma_f16(td, ba + static_cast<uint64_t>(((kk >> 2) * L::HALF_Q + (kk & 3) * 32) >> 4),
                     bb + static_cast<uint64_t>(((kk >> 2) * L::HALF_KT + (kk & 3) * 32) >> 4), id_s, kk > 0 ? 1u : 0u);
          }
          umma_commit(s_full(g));
        };
        auto issue_pv = [&](int g, int st, int j, bool last) {
          tc_fence_after_sync();
          const uint64_t bb = dv + static_cast<uint64_t>((st * L::KT_BYTES) >> 4);
          const uint32_t tt = tmem + g * L::TMEM_TILE;
#pragma unroll
          for (int kk = 0; kk < kKeys / 16; ++kk) {
            umma_f16_tmem_a(tt + L::TMEM_O, tt + L::TMEM_S + kk * 8, bb + static_cast<uint64_t>((kk * 2048) >> 4), id_o,
                            (j > 0 || kk > 0) ? 1u : 0u);
          }
          if (last) umma_commit(pv_done(g));   // the epilogue's wait: the item's last PV of tile g
        };
        uint32_t tc = 0, itc = 0;   // steps, items
        int sk = 0, sv = 0;           // K / V ring stages of the next tile
        uint32_t pk = 0, pv = 0;      // and the phase parity of their full barriers
        bool ok = true;
        uint32_t use = 0;   // ring reads
        Item it;
        int kc;
        auto next = [&]() -> int {
          if (!ring_wait(use)) return -2;
          const int kk = ring_get(use, it);
          ring_release(use);
          ++use;
          return kk;
        };
        while (ok && (kc = next()) >= 0) {
          ok = wait1(k_full(sk), pk);
          for (int g = 0; g < NT && ok; ++g) {
            if (!(ok = wait1(q_full(g), itc & 1))) break;
            issue_s(g, sk);
            if (it.nkt == 1) umma_commit(q_empty(g));
          }
          if (!ok) break;
          for (int j = 0; j < it.nkt; ++j, ++tc) {
            const bool more = j + 1 < it.nkt;
            if (++sk == kStagesK) { sk = 0; pk ^= 1u; }   // K tile j + 1 (the next item's first after the last)
            if (!(ok = wait1(v_full(sv), pv))) break;
            const int pb = it.c >> 4;
            if ((it.c & 15) && pb / kBlocksPerTile == j) {
              const uint32_t vbase = sV + sv * L::KT_BYTES;
              const int r0 = it.c & 15;
              for (int idx = 0; idx < (16 - r0) * NBOX * 8; ++idx) {
                const int row = (pb % kBlocksPerTile) * 16 + r0 + idx / (NBOX * 8);
                const int rem = idx % (NBOX * 8);
                const uint32_t addr = vbase + (rem >> 3) * L::HALF_KT + row * 128 + ((rem & 7) << 4);
                asm volatile("st.shared.v4.b32 [%0], {%1,%1,%1,%1};" ::"r"(addr), "r"(0u) : "memory");
              }
              fence_proxy_async_smem();
            }
            for (int g = 0; g < NT; ++g) {
              if (!(ok = wait1(p_full(g), tc & 1) && (j > 0 || itc == 0 || wait1(o_free(g), (itc - 1) & 1))))
                break;
              issue_pv(g, sv, j, !more);
              if (more) {
                if (g == 0 && !(ok = wait1(k_full(sk), pk))) break;
                issue_s(g, sk);
                if (j + 2 == it.nkt) umma_commit(q_empty(g));
              }
            }
            if (!ok) break;
            if (++sv == kStagesV) { sv = 0; pv ^= 1u; }
          }
          ++itc;
        }
        if (kc == -2) ok = false;
        if (!ok) abort_sh = 1;
        umma_commit(mma_final(0));
        mbar_wait_bounded(mma_final(0), 0, 100000000ull);
      }
      __syncwarp();
    } else if (warp == 11) {
      // ---------------------------------------------------------- query loader
      // Q rows of the item's tiles -> shared memory in the 128-byte-swizzled
      // K-major layout: a whole tile by TMA (the 3-D query map), the prompt's
      // last partial tile by cp.async with the rows past the prompt zeroed.
      // bf16 queries for an fp16 pass land on q_raw instead: the tile's
      // softmax threads convert them in place and complete q_full.
      constexpr int CH = D / 8;   // 16-byte chunks per row
      const uint64_t policy_q = l2_policy_evict_first();   // each query tile is read once
      bool ok = true;
      uint32_t itc = 0;
      uint32_t tma_uses[2] = {0u, 0u};   // q_raw phases this warp started (convert mode)
      // The schedule: lane 0 takes item indices from the global counter
      // (skipping items without work) and publishes them into the ring, each
      // once the Q tiles of the item before it are on their way; -1 once the
      // counter has run out.
      uint32_t pub = 0;   // indices published
      // CTA b's first item is item b (the counter starts past the grid), so
      // the first tiles need no round trip to the counter
      bool first = true;
      auto fetch = [&](Item& x) -> int {
        for (;;) {
          const int kk = first ? static_cast<int>(blockIdx.x) : atomicAdd(a.sched, 1) + static_cast<int>(gridDim.x);
          first = false;
          if (kk >= n_items) return -1;
          if (item_at(kk, x)) return kk;
        }
      };
      auto publish = [&](int kk, const Item& x) -> bool {
        const int i = static_cast<int>(pub % kRing);
        if (pub >= kRing && (abort_sh || !mbar_wait_bounded(item_empty(i), ((pub / kRing) - 1) & 1))) return false;
        volatile int* e = ring + kRingEntry * i;
        e[0] = kk;
        e[1] = x.s;
        e[2] = x.h;
        e[3] = x.t;
        e[4] = x.q0;
        e[5] = x.n;
        e[6] = x.c;
        e[7] = x.nkt;
        mbar_arrive(item_full(i));   // release: the readers' acquiring wait sees the entry
        ++pub;
        return true;
      };
      // lane 0 takes and publishes the next item; the warp shares it
      auto fetch_publish = [&](int& kk, Item& x) -> bool {
        int ok1 = 1;
        kk = -1;
        if (lane == 0) {
          kk = fetch(x);
          ok1 = publish(kk, x) ? 1 : 0;
        }
        kk = __shfl_sync(0xffffffffu, kk, 0);
        x.s = __shfl_sync(0xffffffffu, x.s, 0);
        x.h = __shfl_sync(0xffffffffu, x.h, 0);
        x.t = __shfl_sync(0xffffffffu, x.t, 0);
        x.q0 = __shfl_sync(0xffffffffu, x.q0, 0);
        x.n = __shfl_sync(0xffffffffu, x.n, 0);
        x.c = __shfl_sync(0xffffffffu, x.c, 0);
        x.nkt = __shfl_sync(0xffffffffu, x.nkt, 0);
        return __shfl_sync(0xffffffffu, ok1, 0) != 0;
      };
      Item it{}, nx{};
      int kc;
      ok = fetch_publish(kc, it);
      while (ok && kc >= 0) {
        for (int g = 0; g < NT && ok; ++g) {
          // the previous item's S products of this tile (its last reads of
          // Q_g) have completed
          if (itc > 0) {
            ok = !abort_sh && mbar_wait_bounded(q_empty(g), (itc - 1) & 1);
            if (!__all_sync(0xffffffffu, ok)) {
              ok = false;
              break;
            }
          }
          const uint32_t qbase = sQ + g * L::Q_BYTES;
          if ((it.t + 1) * kRows <= it.n) {
            // a whole tile: NBOX boxes of 128 rows x 64 columns, by TMA
            if (lane == 0) {
              const uint32_t bar = kCvtQ ? q_raw(g) : q_full(g);
              mbar_arrive_expect_tx(bar, L::Q_BYTES);
              for (int h = 0; h < NBOX; ++h)
                tma_load_3d(qbase + h * L::HALF_Q, &qmap, h * 64, it.h + g, it.q0 + it.t * kRows, bar, policy_q);
            }
            __syncwarp();
          } else {
            // the prompt's last, partial tile (whose rows past the prompt may
            // lie past the caller's buffer): cp.async of the rows that exist
            const TA* qh = static_cast<const TA*>(a.q) + static_cast<size_t>(it.h + g) * D;
            for (int idx = lane; idx < kRows * CH; idx += 32) {
              const int r = idx / CH;
              const int cc = idx - r * CH;
              const int lr = it.t * kRows + r;
              const bool in = lr < it.n;
              const TA* src = in ? qh + (static_cast<size_t>(it.q0) + lr) * H * D + cc * 8 : qh;
              const uint32_t dst = qbase + (cc >> 3) * L::HALF_Q + r * 128 + (((cc & 7) ^ (r & 7)) << 4);
              cp_async_16(dst, src, in ? 16u : 0u);
            }
            cp_async_wait_all();
            if constexpr (!kCvtQ) fence_proxy_async_smem();   // the MMAs (async proxy) read what these copies wrote
            __syncwarp();
            if (lane == 0) mbar_arrive(kCvtQ ? q_raw(g) : q_full(g));
          }
          if constexpr (kCvtQ) ++tma_uses[g];
        }
        if (!ok) break;
        ++itc;
        // the next index once this item's Q tiles are on their way (the
        // counter's round trip stays off their path; the readers want it
        // only at this item's end)
        int kn;
        if (!(ok = fetch_publish(kn, nx))) break;
        kc = kn;
        it = nx;
      }
      if (!ok) abort_sh = 1;
      if (kCvtQ && lane == 0) {
        // the last copy of each tile may still be in flight when the softmax
        // warps have stopped waiting for it (an abort): let it land
        for (int g = 0; g < NT; ++g)
          if (tma_uses[g] > 0) mbar_wait_bounded(q_raw(g), (tma_uses[g] - 1) & 1u, 100000000ull);
      }
    }
    teardown();
  } else if (warp < 4 || paired) {
    asm volatile("setmaxnreg.inc.sync.aligned.u32 %0;" ::"n"(kRegsSoftmax));
    // ------------------------------------------------- softmax + epilogue of tile g
    const int g = warp >> 2;
    const int r = threadIdx.x & 127;   // query row of the tile (tensor-memory lane)
    const uint32_t tt = tmem + g * L::TMEM_TILE;
    const uint32_t lane_base = static_cast<uint32_t>((warp & 3) * 32) << 16;
    const uint32_t tO = tt + L::TMEM_O + lane_base;
    const uint32_t tbuf = tt + L::TMEM_S + lane_base;
    // scale > 0 (the usual case): the max is taken on the raw scores and the
    // scale folds into one FMA per element; otherwise scale first.
    const bool pos_scale = a.scale_log2 > 0.f;
    const float sc = pos_scale ? a.scale_log2 : 1.f;   // p = 2^(x*sc - mu) on raw scores x
    uint32_t tc = 0, itc = 0;
    uint32_t kvc = 0;   // K/V tiles of the items before this one
    // the last tile's softmax hands the K and V stages back to the producers:
    // S_g(j) of the last tile completes after every earlier product of the
    // single issuing thread (PV(j - 1) of both tiles included)
    const bool releaser = g == NT - 1 && (warp & 3) == 0 && lane == 0;
    const bool out32 = (reinterpret_cast<uintptr_t>(a.out) & 31u) == 0;   // rows of D >= 64 elements start 32-byte aligned
    // bf16 queries for an fp16 pass: the tile's 128 threads convert its Q
    // tile in place once it has landed (q_raw) and complete q_full -- the
    // first item's before its loop, each next item's while the current
    // item's last PV runs, so the next S can start during the epilogue.  A
    // bf16 exponent field of 143 or more (|x| >= 2^16, inf, NaN) carries
    // (256 - 143) into its half's top bit, which `range` collects; such
    // values saturate to +-65504.
    uint32_t range = 0;
    auto convert_q = [&](uint32_t use) -> bool {
      const bool landed = !abort_sh && mbar_wait_bounded(q_raw(g), use & 1u);
      if (!__all_sync(0xffffffffu, landed)) return false;
      const uint32_t qbase = sQ + g * L::Q_BYTES;
#pragma unroll 4
      for (int off = r * 16; off < L::Q_BYTES; off += kRows * 16) {
        const uint4 v = lds128(qbase + off);
        const uint32_t w[4] = {v.x, v.y, v.z, v.w};
        uint32_t o[4];
#pragma unroll
        for (int e = 0; e < 4; ++e) {
          range |= (w[e] & 0x7f807f80u) + 0x38803880u;
          asm("cvt.rn.satfinite.f16x2.f32 %0, %1, %2;"
              : "=r"(o[e])
              : "f"(__uint_as_float(w[e] & 0xffff0000u)), "f"(__uint_as_float(w[e] << 16)));
        }
        sts128(qbase + off, o[0], o[1], o[2], o[3]);
      }
      fence_proxy_async_smem();   // the MMAs (async proxy) read what these threads wrote
      __syncwarp();
      if (lane == 0) mbar_arrive(q_full(g));
      return true;
    };
    bool ok = true;
    uint32_t use = 0;   // ring reads
    // the next item from the ring, read by the whole warp
    auto next = [&](Item& x) -> int {
      if (!__all_sync(0xffffffffu, ring_wait(use))) return -2;
      const int kk = ring_get(use, x);
      __syncwarp();
      if (lane == 0) ring_release(use);
      ++use;
      return kk;
    };
    Item it, nx;
    int kc = next(it);
    bool have = kc >= 0;
    if constexpr (kCvtQ) {
      if (have) ok = convert_q(0);
    }
    while (ok && have) {
      const int pos = it.c - it.n + it.t * kRows + r;                    // causal limit of this row
      const int warp_pos_min = it.c - it.n + it.t * kRows + (warp & 3) * 32;
      float m_used = -INFINITY;   // reference max of this row (log2 domain)
      float l = 0.f;              // sum of 2^(x - m_used)
      for (int j = 0; j < it.nkt; ++j, ++tc) {
        ok = !abort_sh && mbar_wait_bounded(s_full(g), tc & 1);
        if (!__all_sync(0xffffffffu, ok)) {
          ok = false;
          break;
        }
        tc_fence_after_sync();
        if (releaser) {
          mbar_arrive(k_empty(static_cast<int>((kvc + j) % kStagesK)));
          if (j > 0) mbar_arrive(v_empty(static_cast<int>((kvc + j - 1) % kStagesV)));
        }
        const int key0 = j * kKeys;
        const bool diag = key0 + kKeys - 1 > warp_pos_min;   // a tile on the diagonal: causal mask
        float x[kKeys];
        tmem_ld128(tbuf, x);
        if (!pos_scale) {
#pragma unroll
          for (int i = 0; i < kKeys; ++i) x[i] *= a.scale_log2;
        }
        if (diag) {
          // keys key0 .. key0 + lim are visible to this row: a select per
          // key (the rows of a warp differ, so a branch would diverge)
          const int lim = pos - key0;
#pragma unroll
          for (int i = 0; i < kKeys; ++i) x[i] = i > lim ? -INFINITY : x[i];
        }
        float pm[8];
#pragma unroll
        for (int q = 0; q < 8; ++q) pm[q] = x[q];
#pragma unroll
        for (int i = 8; i < kKeys; i += 8)
#pragma unroll
          for (int q = 0; q < 8; ++q) pm[q] = fmaxf(pm[q], x[i + q]);
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
          // rescale this warp's rows of O: PV_g(j - 1) was issued before S_g(j),
          // so it has completed once S_g(j) has
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
      if (!ok) break;
      // the next item, looked up while this item's last PV runs
      const int kn = next(nx);
      const bool have_next = kn >= 0;
      if constexpr (kCvtQ) {
        if (have_next && !(ok = convert_q(itc + 1))) break;
      }
      // epilogue: once the item's last PV has completed, O / l -> out
      ok = !abort_sh && mbar_wait_bounded(pv_done(g), itc & 1);
      if (!__all_sync(0xffffffffu, ok)) {
        ok = false;
        break;
      }
      if (releaser) mbar_arrive(v_empty(static_cast<int>((kvc + it.nkt - 1) % kStagesV)));
      kvc += it.nkt;
      ++itc;
      tc_fence_after_sync();
      const float inv = l > 0.f ? 1.f / l : 0.f;
      const int lr = it.t * kRows + r;
      TA* orow = static_cast<TA*>(a.out) + ((static_cast<size_t>(it.q0) + lr) * H + it.h + g) * D;
#pragma unroll
      for (int cc = 0; cc < D / 32; ++cc) {
        float o[32];
        tmem_ld32(tO + cc * 32, o);
        if (lr < it.n) {
          uint32_t w[16];
#pragma unroll
          for (int e = 0; e < 16; ++e) w[e] = Mma<TA>::pack(o[2 * e] * inv, o[2 * e + 1] * inv);
          if (out32) {
            // whole 32-byte sectors per store (the rows are 32-byte aligned when out is)
#pragma unroll
            for (int e = 0; e < 2; ++e)
              asm volatile("st.global.v8.b32 [%0], {%1,%2,%3,%4,%5,%6,%7,%8};" ::"l"(orow + cc * 32 + 16 * e),
                           "r"(w[8 * e]), "r"(w[8 * e + 1]), "r"(w[8 * e + 2]), "r"(w[8 * e + 3]), "r"(w[8 * e + 4]),
                           "r"(w[8 * e + 5]), "r"(w[8 * e + 6]), "r"(w[8 * e + 7])
                           : "memory");
          } else {
#pragma unroll
            for (int e = 0; e < 4; ++e)
              reinterpret_cast<uint4*>(orow + cc * 32)[e] = make_uint4(w[4 * e], w[4 * e + 1], w[4 * e + 2], w[4 * e + 3]);
          }
        }
      }
      tc_fence_before_sync();
      __syncwarp();
      if (lane == 0) mbar_arrive(o_free(g));
      kc = kn;
      have = have_next;
      it = nx;
    }
    if (kc == -2) ok = false;
    if (!ok) abort_sh = 1;
    if (kCvtQ && (range & 0x80008000u)) flag_status(a.status, PA_DEV_RANGE);
    teardown();
    if (threadIdx.x == 0 && abort_sh) flag_status(a.status, PA_DEV_WAIT_TIMEOUT);
    if (threadIdx.x == 0) {
      // the last CTA to finish returns the launch's counters to zero for the
      // next launch that draws the same slot (every CTA's last take of an
      // item index precedes its teardown, and so its count here)
      __threadfence();
      if (atomicAdd(a.sched + 1, 1) == static_cast<int>(gridDim.x) - 1) {
        a.sched[0] = 0;
        a.sched[1] = 0;
        __threadfence();
      }
    }
    if (warp == 0) {
      tc_fence_after_sync();
      tmem_dealloc(tmem, kTmemCols);
    }
  } else {
    // tile B's softmax warps when the query group is odd (no tile B): idle
    asm volatile("setmaxnreg.inc.sync.aligned.u32 %0;" ::"n"(kRegsSoftmax));
    teardown();
  }
}

namespace {
template <typename T, typename TA, int D>
cudaError_t launch_umma_t(const PrefillArgs& a, const CUtensorMap& kmap, const CUtensorMap& vmap,
                          const CUtensorMap& qmap, cudaStream_t stream) {
  const int smem = UmmaLayout<D>::SMEM + 1024;
  auto kern = prefill_umma_kernel<T, TA, D>;
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
  if (e != cudaSuccess) return e;
  // persistent: one CTA per SM, or fewer when there are fewer items
  int sms = device_sm_count();
  if (sms <= 0) sms = 152;
  const int nt = (a.num_q_heads / a.num_kv_heads) % 2 == 0 ? 2 : 1;
  const long long items = static_cast<long long>((a.max_q_len + kRows - 1) / kRows) * (a.num_q_heads / nt) *
                          a.num_seqs;
  const long long ctas = items < sms ? items : sms;
  if (ctas <= 0) return cudaSuccess;
  return launch_pdl(kern, dim3(static_cast<unsigned>(ctas)), dim3(kThreads), smem, stream, kmap, vmap, qmap, a);
}

template <typename T, typename TA>
cudaError_t launch_umma_d(const PrefillArgs& a, const CUtensorMap& kmap, const CUtensorMap& vmap,
                          const CUtensorMap& qmap, cudaStream_t stream) {
  return a.head_dim == 128 ? launch_umma_t<T, TA, 128>(a, kmap, vmap, qmap, stream)
                           : launch_umma_t<T, TA, 64>(a, kmap, vmap, qmap, stream);
}
}  // namespace

cudaError_t launch_prefill_umma(const PrefillArgs& a, int dtype, int act_dtype, const CUtensorMap& kmap,
                                const CUtensorMap& vmap, const CUtensorMap& qmap, cudaStream_t stream) {
  if (dtype == PA_BF16) return launch_umma_d<__nv_bfloat16, __nv_bfloat16>(a, kmap, vmap, qmap, stream);
  if (act_dtype == PA_BF16) return launch_umma_d<__half, __nv_bfloat16>(a, kmap, vmap, qmap, stream);
  return launch_umma_d<__half, __half>(a, kmap, vmap, qmap, stream);
}

}  // namespace pa
