// verify_umma.cu -- attention of the verification pass of speculative decoding
// (q_len query positions per sequence, causal over the paged cache) on the
// 5th-generation tensor cores, as one persistent, stream-K balanced launch.
//
// The target model checks K drafted tokens in one forward pass ("LLM
// Inference Server", Batched Scheduling & Speculative Decoding: K = 4): query
// i of a sequence with context c sits at position c - q_len + i and sees keys
// 0 .. c - q_len + i.  Per KV head the query columns are the G heads of the
// group at every position (column x = i * G + h): NC = 16 or 32 MMA columns,
// the unused ones zero, of which the softmax works on CU (the used ones rounded
// up to 8).  Every column of a (sequence, KV head) reads the same
// K/V, so the work is two thin matrix products per 128-token tile -- scores
// S^T = K q^T (M = 128 tokens, N = NC, K = D) and O^T += V^T P (M = D,
// N = NC, K = 128 tokens) -- with the softmax between them.
//
// Work split (stream-K): the (sequence, KV head, 128-token tile) triples, in
// sequence-major order, are cut into one contiguous range per CTA of equal
// cost (at least `part_blocks / 8` tiles), so every SM finishes at the same
// time whatever the context lengths; a run's cost counts its tiles and the
// fixed cost of starting it.  A range covers whole or partial (sequence, KV
// head) runs, "segments"; a (sequence, KV head) split over several CTAs leaves
// one normalised partial per segment and the CTA that finishes its segment
// last merges them by log-sum-exp.
//
// One CTA per SM, twelve warps with fixed roles:
//   warps 0-3  softmax: thread t owns token row t of S^T (tensor memory lane
//              t).  The softmax reference of each column is shared by the CTA
//              and raised lazily (only when a score exceeds it by 2^8; a CTA-
//              wide vote decides, a transpose reduction gives the column
//              maxima).  Each thread writes its row of P (the second
//              product's B operand, MN-major, 64- or 32-byte swizzle) to shared
//              memory with 16-byte stores; a raise rescales O^T in tensor memory.
//   warps 4-7  epilogue: thread d owns head-dim row d of O^T.  It normalises
//              and stores each finished segment and runs the split-K merge;
//              none of this holds up the tiles of the next segments.
//   warps 8/10 TMA producers of K tiles (2 stages) and V tiles (3 stages) of
//              8 pool blocks through the block table; blocks past the context
//              or with an id outside the pool are read as zeros.  The V warp
//              also stages each segment's q.
//   warps 9/11 MMA issuers: S^T of tile j (warp 9) and O^T += V^T P of tile j
//              (warp 11), so the scores of the next tile are computed while the
//              softmax of this one runs.
// Tensor memory: two S^T buffers and three O^T buffers of NC columns (O^T
// rotates by segment so the epilogues of the last two overlap the next).
//
// Stale pool rows past a sequence's last token are zeroed in shared memory
// before the second product reads them (their weight is 0, and 0 * NaN is
// not).  Every wait is bounded; a timeout sets PA_DEV_WAIT_TIMEOUT and the
// roles leave their loops together.
#include <type_traits>

#include "decode_merge.cuh"
#include "pa_common.cuh"
#include "pa_internal.h"

namespace pa {

namespace {

constexpr int kTok = 128;                      // tokens per tile (MMA M of S^T)
constexpr int kTileBlocks = kTok / kBlock;     // 8 pool blocks
constexpr int kDim = 128;                      // head dim (MMA M of O^T)
constexpr int kStrip = kTok * 128;             // one 64-column strip of a K or V tile
constexpr int kTileBytes = 2 * kStrip;         // 32 KB
constexpr int kKStages = 2;
constexpr int kVStages = 3;
constexpr int kUThreads = 384;
constexpr float kLazyU = 8.f;                  // log2 headroom of the softmax reference

template <int NC>
struct VLayout {
  static constexpr int QSTRIP = NC * 128;      // one 64-column strip of q (NC rows)
  static constexpr int QBYTES = 2 * QSTRIP;
  static constexpr int PBYTES = kTok * NC * 2; // P: 128 token rows of NC columns (two buffers)
  static constexpr int K_OFF = 0;
  static constexpr int V_OFF = K_OFF + kKStages * kTileBytes;
  static constexpr int Q_OFF = V_OFF + kVStages * kTileBytes;
  static constexpr int P_OFF = Q_OFF + 2 * QBYTES;
  static constexpr int SMEM = P_OFF + 2 * PBYTES;
  static constexpr uint32_t TMEM_COLS = NC == 32 ? 256 : 128;   // S^T x2, O^T x3 (a power of two)
};

template <typename T>
__device__ __forceinline__ uint16_t bits16(float x);
template <>
__device__ __forceinline__ uint16_t bits16<__nv_bfloat16>(float x) {
  return __bfloat16_as_ushort(__float2bfloat16_rn(x));
}
template <>
__device__ __forceinline__ uint16_t bits16<__half>(float x) {
  return __half_as_ushort(__float2half_rn(x));
}

__device__ __forceinline__ bool cta_any(int barrier_id, bool v) {
  uint32_t r;
  asm volatile(
      "{\n\t.reg .pred p, q;\n\t"
      "setp.ne.u32 p, %1, 0;\n\t"
      "bar.red.or.pred q, %2, 128, p;\n\t"
      "selp.u32 %0, 1, 0, q;\n\t}"
      : "=r"(r)
      : "r"(v ? 1u : 0u), "r"(barrier_id)
      : "memory");
  return r != 0;
}

// Bounded wait for roles whose waits are long and off the critical path: between
// polls the thread naps ~0.1 us, so it takes few issue slots from the softmax warps
// and wakes at most that late.
__device__ __forceinline__ bool mbar_wait_idle(uint32_t bar, uint32_t parity, uint64_t limit_ns = 1000000000ull) {
  if (mbar_try_wait(bar, parity)) return true;
  const uint64_t t0 = global_timer_ns();
  while (true) {
    __nanosleep(100);
    if (mbar_try_wait(bar, parity)) return true;
    if (global_timer_ns() - t0 > limit_ns) return false;
  }
}

__device__ __forceinline__ void group_sync(int barrier_id) {
  asm volatile("bar.sync %0, 128;" ::"r"(barrier_id) : "memory");
}

// Shared-memory descriptor of an MN-major operand whose MN extent is one swizzle
// atom (NC = 32: 64-byte rows, 64-byte swizzle; NC = 16: 32-byte rows, 32-byte
// swizzle); sbo = bytes between atoms of 8 rows along K.
template <int NC>
__device__ __forceinline__ uint64_t umma_desc_mn_t(uint32_t smem_addr, uint32_t sbo_bytes) {
  uint64_t d = 0;
  d |= static_cast<uint64_t>((smem_addr >> 4) & 0x3FFFu);
  d |= static_cast<uint64_t>((sbo_bytes >> 4) & 0x3FFFu) << 16;   // leading offset: unused for one atom
  d |= static_cast<uint64_t>((sbo_bytes >> 4) & 0x3FFFu) << 32;
  d |= static_cast<uint64_t>(1) << 46;                            // descriptor version
  d |= static_cast<uint64_t>(NC == 32 ? 4 : 6) << 61;             // 64- or 32-byte swizzle
  return d;
}

// The first CU (8, 16, 24 or 32) fp32 columns of this thread's TMEM lane.
__device__ __forceinline__ void tmem_ld8(uint32_t taddr, float* v) {
  uint32_t r[8];
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x8.b32 {%0,%1,%2,%3,%4,%5,%6,%7}, [%8];\n\t"
      "tcgen05.wait::ld.sync.aligned;"
      : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7])
      : "r"(taddr)
      : "memory");
#pragma unroll
  for (int i = 0; i < 8; ++i) v[i] = __uint_as_float(r[i]);
}
template <int CU>
__device__ __forceinline__ void load_cols(uint32_t taddr, float* v) {
  if constexpr (CU == 32) {
    tmem_ld32(taddr, v);
  } else if constexpr (CU == 24) {
    tmem_ld16(taddr, v);
    tmem_ld8(taddr + 16, v + 16);
  } else if constexpr (CU == 16) {
    tmem_ld16(taddr, v);
  } else {
    tmem_ld8(taddr, v);
  }
}

// Transpose reduction over a warp: v[0..CU) per lane in; lane x (x < CU)
// gets the reduction over all 32 lanes of column x.
template <int CU, bool MAX>
__device__ __forceinline__ float warp_columns(const float* v, int lane) {
  constexpr int P2 = CU <= 8 ? 8 : CU <= 16 ? 16 : 32;
  float w[P2];
#pragma unroll
  for (int k = 0; k < P2; ++k) w[k] = k < CU ? v[k] : (MAX ? -INFINITY : 0.f);
#pragma unroll
  for (int off = 16; off >= P2; off >>= 1)   // fold the lanes above P2
#pragma unroll
    for (int k = 0; k < P2; ++k) {
      const float o = __shfl_xor_sync(0xffffffffu, w[k], off);
      w[k] = MAX ? fmaxf(w[k], o) : w[k] + o;
    }
#pragma unroll
  for (int off = P2 / 2; off >= 1; off >>= 1) {
    const bool hi = (lane & off) != 0;
#pragma unroll
    for (int k = 0; k < off; ++k) {
      const float send = hi ? w[k] : w[k + off];
      const float keep = hi ? w[k + off] : w[k];
      const float o = __shfl_xor_sync(0xffffffffu, send, off);
      w[k] = MAX ? fmaxf(keep, o) : keep + o;
    }
  }
  return w[0];
}

// The CTA's share of the global tile order: sequence by sequence, KV head by
// KV head, tile by tile.  All roles walk it identically.
struct Segment {
  int s, kvh, j0, ntiles;   // tiles j0 .. j0 + ntiles - 1 of (s, kvh)
  int ctx, nt;              // context and tile count of sequence s
  int n_parts, part;        // segments of (s, kvh) over all CTAs, and this one's index
};

// The split balances cost, not tiles: a (sequence, KV head) run of nt tiles
// weighs nt * kUnitsTile + kUnitsSeg units (a tile, plus the fixed cost of a
// segment: its first scores raise every reference, its statistics and outputs
// are written once).  Tile j of a run at unit b sits at unit b + kUnitsTile * j
// and belongs to the CTA whose range of units holds that point; ranges are at
// least kUnitsTile long, so every CTA between a run's first and last owner holds
// one of its tiles.
constexpr int kUnitsTile = 4;
constexpr int kUnitsSeg = 16;

struct Walk {
  int s, kvh, j, ctx, nt;
  long long ibase;          // unit of the current run's first tile
  long long x1;             // end of this CTA's range of units
};

__device__ __forceinline__ long long owner_of(long long x, long long V, int geff) {
  return ((x + 1) * geff - 1) / V;
}

__device__ __forceinline__ int tiles_of(int ctx) { return (ctx + kTok - 1) / kTok; }
__device__ __forceinline__ long long run_units(int nt) {
  return nt > 0 ? static_cast<long long>(kUnitsTile) * nt + kUnitsSeg : 0;
}

// Contexts of the CTA's first kCtxCache sequences, cached in shared memory: every
// role walks the same sequences, and a global load per new sequence would stall it.
constexpr int kCtxCache = 64;

__device__ __forceinline__ int walk_context(const DecodeArgs& a, const int* cache, int s0, int s) {
  return s - s0 < kCtxCache ? cache[s - s0] : checked_context(a, s, false);
}

// Next segment of the walk; false when the CTA's range is done.
__device__ __forceinline__ bool next_segment(const DecodeArgs& a, Walk& w, long long V, int geff, Segment& g,
                                             const int* cache, int s0) {
  while (w.nt == 0 || w.j >= w.nt) {   // the walk never rests on an empty or finished run
    if (w.nt > 0 && w.j >= w.nt) {
      w.j = 0;
      w.ibase += run_units(w.nt);
      if (++w.kvh < a.num_kv_heads) continue;
    }
    w.kvh = 0;
    w.j = 0;
    ++w.s;
    if (w.s >= a.num_seqs) return false;
    w.ctx = walk_context(a, cache, s0, w.s);
    w.nt = tiles_of(w.ctx);
  }
  const long long r = w.x1 - w.ibase;   // this CTA's tiles of the run: kUnitsTile * j < r
  if (r <= 0) return false;
  const int jend = static_cast<int>(min(static_cast<long long>(w.nt), (r + kUnitsTile - 1) / kUnitsTile));
  if (jend <= w.j) return false;
  g.s = w.s;
  g.kvh = w.kvh;
  g.j0 = w.j;
  g.ctx = w.ctx;
  g.nt = w.nt;
  g.ntiles = jend - w.j;
  const long long c0 = owner_of(w.ibase, V, geff);
  const long long c1 = owner_of(w.ibase + static_cast<long long>(kUnitsTile) * (w.nt - 1), V, geff);
  g.n_parts = static_cast<int>(c1 - c0 + 1);
  g.part = static_cast<int>(blockIdx.x - c0);
  w.j = jend;
  return true;
}

}  // namespace

template <typename T, int NC, int CU>
__global__ void __launch_bounds__(kUThreads, 1)
verify_umma_kernel(const __grid_constant__ CUtensorMap kmap, const __grid_constant__ CUtensorMap vmap,
                   const DecodeArgs a) {
  using L = VLayout<NC>;
  constexpr bool kBf16 = !std::is_same<T, __half>::value;
  constexpr int D = kDim;

  extern __shared__ uint8_t smem_raw[];
  // kfull[3] kempty[3] vfull[3] vempty[3] qfull[2] qempty[2] sfull[2] sfree[2]
  // pfull[2] pfree[2] ofull[3] ofree[3] stfull[3] stfree[3] final
  __shared__ __align__(8) uint64_t bars[37];
  __shared__ float red_sh[4][NC];              // column maxima of a raise, per softmax warp
  // The CTA's column references, alternating by raise (-inf while a column has none).
  __shared__ __align__(16) float mu_sh[2][NC];
  __shared__ float st_l[3][4][NC];             // per segment: column sums of each softmax warp
  __shared__ float st_m[3][NC];                // per segment: column references
  __shared__ long long walk_sh[3];             // first run's unit, end of the range, total units
  __shared__ int walk_i[4];                    // s, kvh, j, geff
  __shared__ int ctx_sh[kCtxCache];            // contexts of sequences walk_i[0] ...
  __shared__ uint32_t tmem_base_sh;
  __shared__ volatile int abort_sh;
  __shared__ int last_sh;

  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                             ~static_cast<uintptr_t>(1023));
  const uint32_t sK = smem_u32(smem) + L::K_OFF;
  const uint32_t sV = smem_u32(smem) + L::V_OFF;
  const uint32_t sQ = smem_u32(smem) + L::Q_OFF;
  const uint32_t sP = smem_u32(smem) + L::P_OFF;
  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const int G = a.num_q_heads / a.num_kv_heads;
  const int NQ = G * a.q_len;
  const int H = a.num_kv_heads;

  const uint32_t bar0 = smem_u32(&bars[0]);
  auto kfull = [&](int i) { return bar0 + 8u * i; };
  auto kempty = [&](int i) { return bar0 + 24u + 8u * i; };
  auto vfull = [&](int i) { return bar0 + 48u + 8u * i; };
  auto vempty = [&](int i) { return bar0 + 72u + 8u * i; };
  auto qfull = [&](int i) { return bar0 + 96u + 8u * i; };
  auto qempty = [&](int i) { return bar0 + 112u + 8u * i; };
  auto sfull = [&](int i) { return bar0 + 128u + 8u * i; };
  auto sfree = [&](int i) { return bar0 + 144u + 8u * i; };
  auto pfull = [&](int i) { return bar0 + 160u + 8u * i; };
  auto pfree = [&](int i) { return bar0 + 176u + 8u * i; };
  auto ofull = [&](int i) { return bar0 + 192u + 8u * i; };
  auto ofree = [&](int i) { return bar0 + 216u + 8u * i; };
  auto stfull = [&](int i) { return bar0 + 240u + 8u * i; };
  auto stfree = [&](int i) { return bar0 + 264u + 8u * i; };
  const uint32_t final_bar = bar0 + 288u;

  grid_dependency_wait();   // the cache and the queries come from the kernels before us

  if (threadIdx.x == 0) {
    for (int i = 0; i < kKStages; ++i) {
      mbar_init(kfull(i), 1);
      mbar_init(kempty(i), 1);
    }
    for (int i = 0; i < kVStages; ++i) {
      mbar_init(vfull(i), 1);
      mbar_init(vempty(i), 1);
    }
    for (int i = 0; i < 2; ++i) {
      mbar_init(qfull(i), 1);
      mbar_init(qempty(i), 1);
      mbar_init(sfull(i), 1);
      mbar_init(sfree(i), 4);
      mbar_init(pfull(i), 4);
      mbar_init(pfree(i), 1);
    }
    for (int i = 0; i < 3; ++i) {
      mbar_init(ofull(i), 1);
      mbar_init(ofree(i), 4);
      mbar_init(stfull(i), 4);
      mbar_init(stfree(i), 4);
    }
    mbar_init(final_bar, 2);
    fence_barrier_init();
    abort_sh = 0;
  }
  // ---- the CTA's range of the global tile order (warp 8) ----------------------
  if (warp == 8) {
    long long usum = 0;   // units of one KV head over all sequences
    for (int s0 = 0; s0 < a.num_seqs; s0 += 32) {
      const int s = s0 + lane;
      long long v = s < a.num_seqs ? run_units(tiles_of(checked_context(a, s, blockIdx.x == 0))) : 0;
#pragma unroll
      for (int m = 1; m < 32; m <<= 1) v += __shfl_xor_sync(0xffffffffu, v, m);
      usum += v;
    }
    const long long vtot = usum * H;
    const long long lmin = a.part_blocks >= kTileBlocks ? a.part_blocks / kTileBlocks : 1;
    long long ge = vtot / (lmin * kUnitsTile);
    ge = ge < 1 ? 1 : ge;
    const int geff = static_cast<int>(ge < gridDim.x ? ge : gridDim.x);
    const long long c = blockIdx.x;
    const long long x0 = c < geff ? c * vtot / geff : vtot;
    const long long x1 = c < geff ? (c + 1) * vtot / geff : vtot;
    // locate x0: sequence s whose H runs span [pre, pre + H * units(s)) around it
    long long pre = 0;
    int fs = a.num_seqs, fkvh = 0, fj = 0;
    long long fbase = vtot;
    for (int s0 = 0; s0 < a.num_seqs && fs == a.num_seqs; s0 += 32) {
      const int s = s0 + lane;
      const long long u = s < a.num_seqs ? run_units(tiles_of(checked_context(a, s, false))) : 0;
      long long incl = u * H;
#pragma unroll
      for (int m = 1; m < 32; m <<= 1) {
        const long long o = __shfl_up_sync(0xffffffffu, incl, m);
        if (lane >= m) incl += o;
      }
      const long long excl = incl - u * H;
      const bool hit = s < a.num_seqs && u > 0 && pre + excl <= x0 && x0 < pre + incl;
      const unsigned hm = __ballot_sync(0xffffffffu, hit);
      if (hm) {
        const int src = __ffs(hm) - 1;
        const long long b = __shfl_sync(0xffffffffu, pre + excl, src);
        const long long us = __shfl_sync(0xffffffffu, u, src);
        fs = s0 + src;
        const long long off = x0 - b;
        fkvh = static_cast<int>(off / us);
        fbase = b + fkvh * us;
        fj = static_cast<int>((off - fkvh * us + kUnitsTile - 1) / kUnitsTile);   // may pass the run's end
      }
      pre += __shfl_sync(0xffffffffu, incl, 31);
    }
    for (int k = lane; k < kCtxCache; k += 32)
      ctx_sh[k] = fs + k < a.num_seqs ? checked_context(a, fs + k, false) : 0;
    if (lane == 0) {
      walk_sh[0] = fbase;
      walk_sh[1] = x1;
      walk_sh[2] = vtot;
      walk_i[0] = fs;
      walk_i[1] = fkvh;
      walk_i[2] = fj;
      walk_i[3] = geff;
    }
  }
  if (warp == 0) {
    tmem_alloc(smem_u32(&tmem_base_sh), L::TMEM_COLS);
    tmem_relinquish();
  }
  tc_fence_before_sync();
  __syncthreads();
  tc_fence_after_sync();
  const uint32_t tmem = tmem_base_sh;
  const long long vtot = walk_sh[2];
  const int geff = walk_i[3];
  auto make_walk = [&]() {
    Walk w;
    w.s = walk_i[0];
    w.kvh = walk_i[1];
    w.j = walk_i[2];
    w.ibase = walk_sh[0];
    w.x1 = walk_sh[1];
    w.ctx = w.s < a.num_seqs ? ctx_sh[0] : 0;
    w.nt = tiles_of(w.ctx);
    return w;
  };
  auto waitb = [&](uint32_t bar, uint32_t parity) -> bool {
    return !abort_sh && mbar_wait_bounded(bar, parity);
  };
  auto waiti = [&](uint32_t bar, uint32_t parity) -> bool {   // off the critical path: sleep
    return !abort_sh && mbar_wait_idle(bar, parity);
  };
  const uint32_t id_s = umma_idesc_f16(kTok, NC, kBf16, false, false);
  const uint32_t id_o = umma_idesc_f16(kDim, NC, kBf16, true, true);
  const uint32_t tS = tmem;                 // S^T buffers: columns [0, 2 NC)
  const uint32_t tO = tmem + 2 * NC;        // O^T buffers: columns [2 NC, 5 NC), by segment % 3

  if (warp == 8 || warp == 10) {
    // ------------------------------------------------- TMA producers: K (warp 8), V (warp 10)
    // Separate warps, so a K tile is never queued behind a V stage that is still
    // being read: each ring refills as soon as its own stage is released.
    const bool isk = warp == 8;
    const CUtensorMap* map = isk ? &kmap : &vmap;
    const int nst = isk ? kKStages : kVStages;
    const uint32_t ring = isk ? sK : sV;
    if (lane == 0) prefetch_tensormap(map);
    const uint64_t policy = l2_policy_evict_first();
    const int oob_row = a.num_blocks * H * kBlock;   // rows past the pool read as zero
    Walk w = make_walk();
    Segment g;
    int J = 0, I = 0;
    bool ok = true;
    while (ok && next_segment(a, w, vtot, geff, g, ctx_sh, walk_i[0])) {
      if (!isk) {
        // The segment's q, K-major and 128-byte swizzled, once segment I - 2's scores are done.
        // The V warp stages it: its loads stall this warp for a memory latency, which the
        // three V stages absorb, where the two K stages would run dry.
        const int qb = I & 1;
        ok = I < 2 || waiti(qempty(qb), ((I >> 1) - 1) & 1);
        if (!__all_sync(0xffffffffu, ok)) {
          ok = false;
          break;
        }
        const uint32_t qbase = sQ + qb * L::QBYTES;
        const T* qg = static_cast<const T*>(a.q);
        uint4 v[NC / 2];
#pragma unroll
        for (int k = 0; k < NC / 2; ++k) {   // all loads first: one memory latency
          const int idx = lane + 32 * k;
          const int c = idx >> 4;
          v[k] = c < NQ ? __ldg(reinterpret_cast<const uint4*>(qg + query_row(a, g.s, g.kvh, G, c) * D) + (idx & 15))
                        : make_uint4(0u, 0u, 0u, 0u);
        }
#pragma unroll
        for (int k = 0; k < NC / 2; ++k) {
          const int idx = lane + 32 * k;
          const int c = idx >> 4;
          const int cc = idx & 15;
          const uint32_t dst = qbase + (cc >> 3) * L::QSTRIP + c * 128 + (((cc & 7) ^ (c & 7)) << 4);
          asm volatile("st.shared.v4.b32 [%0], {%1,%2,%3,%4};" ::"r"(dst), "r"(v[k].x), "r"(v[k].y), "r"(v[k].z),
                       "r"(v[k].w)
                       : "memory");
        }
        fence_proxy_async_smem();
        __syncwarp();
        if (lane == 0) mbar_arrive(qfull(qb));
      }
      ++I;
      for (int jt = g.j0; jt < g.j0 + g.ntiles; ++jt) {
        // block rows of the tile (looked up before the stage wait, which hides the load)
        int y = oob_row;
        if (lane < kTileBlocks) {
          const int lb = jt * kTileBlocks + lane;
          if (lb * kBlock < g.ctx) {
            const int id = __ldg(a.block_tables + static_cast<size_t>(g.s) * a.max_blocks_per_seq + lb);
            if (id >= 0 && id < a.num_blocks)
              y = (id * H + g.kvh) * kBlock;
            else if (isk)
              flag_status(a.status, PA_DEV_BAD_BLOCK_ID);
          }
        }
        const int yb = __shfl_sync(0xffffffffu, y, lane & (kTileBlocks - 1));
        const int st = J % nst;
        ok = J < nst || waiti(isk ? kempty(st) : vempty(st), ((J / nst) - 1) & 1);
        if (!__all_sync(0xffffffffu, ok)) {
          ok = false;
          break;
        }
        const uint32_t full = isk ? kfull(st) : vfull(st);
        if (lane == 0) mbar_arrive_expect_tx(full, kTileBytes);
        __syncwarp();
        if (lane < 16)
          tma_load_2d(ring + st * kTileBytes + (lane >> 3) * kStrip + (lane & 7) * 2048, map, (lane >> 3) * 64, yb,
                      full, policy);
        ++J;
      }
    }
    if (!ok) abort_sh = 1;
    // every issued copy lands before the CTA may exit (bounded)
    if (lane == 0)
      for (int j = J - nst < 0 ? 0 : J - nst; j < J; ++j)
        mbar_wait_bounded(isk ? kfull(j % nst) : vfull(j % nst), (j / nst) & 1, 100000000ull);
  } else if (warp == 9 || warp == 11) {
    // --------------------------------------------------- MMA issuers: S^T (warp 9), O^T (warp 11)
    // Two issuing warps: issuing stalls while the tensor pipe is busy, and the next
    // tile's scores must not wait behind the previous tile's output product.
    const bool is_s = warp == 9;
    Walk w = make_walk();
    Segment g;
    int J = 0, I = 0;
    bool ok = true;
    while (ok && next_segment(a, w, vtot, geff, g, ctx_sh, walk_i[0])) {
      const int qb = I & 1;
      const int ob = I % 3;
      if (is_s) {
        ok = waitb(qfull(qb), (I >> 1) & 1);
        if (!__all_sync(0xffffffffu, ok)) {
          ok = false;
          break;
        }
      }
      for (int t = 0; t < g.ntiles; ++t, ++J) {
        if (is_s) {
          // S^T_J = K_J q^T once K_J has landed and the softmax has read S_{J-2}
          const int ks = J % kKStages;
          const int sb = J & 1;
          bool k = waitb(kfull(ks), (J / kKStages) & 1);
          if (k && J >= 2) k = waitb(sfree(sb), ((J >> 1) - 1) & 1);
          if (!__all_sync(0xffffffffu, k)) {
            ok = false;
            break;
          }
          tc_fence_after_sync();
          if (lane == 0) {
            const uint64_t da0 = umma_desc_sw128(sK + ks * kTileBytes, 16, 1024);
            const uint64_t db0 = umma_desc_sw128(sQ + qb * L::QBYTES, 16, 1024);
#pragma unroll
            for (int kk = 0; kk < D / 16; ++kk) {   // k-step kk: strip kk / 4, 32 bytes in per step
              const uint64_t da = da0 + static_cast<uint64_t>(((kk >> 2) * kStrip + (kk & 3) * 32) >> 4);
              const uint64_t db = db0 + static_cast<uint64_t>(((kk >> 2) * L::QSTRIP + (kk & 3) * 32) >> 4);
              umma_f16(tS + sb * NC, da, db, id_s, kk > 0 ? 1u : 0u);
            }
            umma_commit(sfull(sb));
            umma_commit(kempty(ks));
            if (t == g.ntiles - 1) umma_commit(qempty(qb));
          }
          __syncwarp();
        } else {
          // O^T += V_J^T P_J once V_J has landed and the softmax has written P_J
          const int vs = J % kVStages;
          const int pb = J & 1;
          bool k = waitb(vfull(vs), (J / kVStages) & 1) && waitb(pfull(pb), (J >> 1) & 1);
          if (k && t == 0 && I >= 3) k = waitb(ofree(ob), ((I / 3) - 1) & 1);
          if (!__all_sync(0xffffffffu, k)) {
            ok = false;
            break;
          }
          tc_fence_after_sync();
          if (lane == 0) {
            const uint64_t da0 = umma_desc_sw128(sV + vs * kTileBytes, kStrip, 1024);
            const uint64_t db0 = umma_desc_mn_t<NC>(sP + pb * L::PBYTES, 8 * NC * 2);
#pragma unroll
            for (int kk = 0; kk < kTok / 16; ++kk) {   // 16 tokens per k-step
              const uint64_t da = da0 + static_cast<uint64_t>((kk * 2048) >> 4);
              const uint64_t db = db0 + static_cast<uint64_t>((kk * 16 * NC * 2) >> 4);
              umma_f16(tO + ob * NC, da, db, id_o, (t == 0 && kk == 0) ? 0u : 1u);
            }
            umma_commit(pfree(pb));
            umma_commit(vempty(vs));
            if (t == g.ntiles - 1) umma_commit(ofull(ob));
          }
          __syncwarp();
        }
      }
      ++I;
    }
    if (!ok) abort_sh = 1;
    // every MMA issued has completed before the CTA tears down (one arrival per issuer)
    if (lane == 0) umma_commit(final_bar);
    mbar_wait_bounded(final_bar, 0, 100000000ull);
  } else if (warp < 4) {
    // ----------------------------------------------------------- softmax warps
    const int t = threadIdx.x;                      // token row of the tile, TMEM lane t
    const uint32_t lane_base = static_cast<uint32_t>(warp * 32) << 16;
    // this row of P in the MN-major B operand: 8 rows of NC columns per swizzle atom
    const uint32_t prow_off = (t >> 3) * (8 * NC * 2) + (t & 7) * (NC * 2);
    const int pswz = NC == 32 ? (t >> 1) & 3 : (t >> 2) & 1;
    Walk w = make_walk();
    Walk wn = make_walk();   // one segment ahead: its first block id is fetched early
    Segment g, gn;
    bool have_n = next_segment(a, wn, vtot, geff, gn, ctx_sh, walk_i[0]);
    auto first_id = [&](const Segment& sg) {
      const int tk = sg.j0 * kTok + t;
      return tk < sg.ctx ? __ldg(a.block_tables + static_cast<size_t>(sg.s) * a.max_blocks_per_seq + tk / kBlock) : 0;
    };
    int id_seg = have_n ? first_id(gn) : 0;
    int J = 0, I = 0, nraise = 0;
    bool ok = true;
    while (next_segment(a, w, vtot, geff, g, ctx_sh, walk_i[0])) {
      int id_next = id_seg;
      have_n = have_n && next_segment(a, wn, vtot, geff, gn, ctx_sh, walk_i[0]);
      if (have_n) id_seg = first_id(gn);
      // per column: the running sum of this row's weights, and the CTA's reference in
      // registers (-inf while there is none; shared memory holds the copy a raise updates)
      float l_part[CU], mu_r[CU];
#pragma unroll
      for (int c = 0; c < CU; ++c) {
        l_part[c] = 0.f;
        mu_r[c] = -INFINITY;
      }
      bool fresh = true;   // no reference yet in this segment
      const int lim0 = g.ctx - a.q_len;   // causal limit of position 0
      bool stop = false;
      // block id of this thread's row, one tile ahead (a row past the context or in a
      // block outside the pool is masked)
      const int32_t* table = a.block_tables + static_cast<size_t>(g.s) * a.max_blocks_per_seq;
      for (int tt = 0; tt < g.ntiles; ++tt) {
        const int jt = g.j0 + tt;
        const int tok = jt * kTok + t;
        const int id = id_next;
        if (tt + 1 < g.ntiles && tok + kTok < g.ctx) id_next = __ldg(table + (tok + kTok) / kBlock);
        const int sb = J & 1;
        bool k = waitb(sfull(sb), (J >> 1) & 1);
        k = __all_sync(0xffffffffu, k);
        if (cta_any(1, !k)) {
          stop = true;
          break;
        }
        tc_fence_after_sync();
        float x[CU];
        load_cols<CU>(tS + sb * NC + lane_base, x);
        tc_fence_before_sync();
        __syncwarp();
        if (lane == 0) mbar_arrive(sfree(sb));
        const bool tok_ok = tok < g.ctx && id >= 0 && id < a.num_blocks;
        const int cmin = tok <= lim0 ? 0 : G * (tok - lim0);   // first column this row may attend
        const bool whole = tok_ok && cmin == 0;                  // every column attends this row
        // x = score in the log2 domain; a raise is due where x passes its reference by more
        // than kLazyU (a factor of 2^8)
        bool need = false;
#pragma unroll
        for (int c = 0; c < CU; ++c) {
          float v = x[c] * a.scale_log2;
          if (!whole) v = (tok_ok && c >= cmin && c < NQ) ? v : -INFINITY;
          x[c] = v;
          need |= v > mu_r[c] + kLazyU;
        }
        if (cta_any(1, need)) {
          // raise: the tile's column maxima over the 128 rows give the new references
          const float r = warp_columns<CU, true>(x, lane);
          if (lane < CU) red_sh[warp][lane] = r;
          group_sync(1);
          const int ob_ = nraise & 1, nb_ = ob_ ^ 1;
          if (warp == 0 && lane < CU) {
            const float mx = fmaxf(fmaxf(red_sh[0][lane], red_sh[1][lane]), fmaxf(red_sh[2][lane], red_sh[3][lane]));
            mu_sh[nb_][lane] = fmaxf(fresh ? -INFINITY : mu_sh[ob_][lane], mx);
          }
          group_sync(1);
          if (!fresh) {   // the first raise of a segment has nothing to rescale
            // 2^(old - new) per column (1 while it had no reference)
            auto alpha = [&](int c) { return mu_r[c] != -INFINITY ? fast_exp2(mu_r[c] - mu_sh[nb_][c]) : 1.f; };
            bool grew = false;
#pragma unroll
            for (int c = 0; c < CU; ++c) grew |= alpha(c) != 1.f;
            if (tt > 0 && grew) {
              // rescale O^T (lane t = head-dim row t) once the previous tile's product is done
              const int pj = J - 1;
              bool k2 = waitb(pfree(pj & 1), (pj >> 1) & 1);
              if (!__all_sync(0xffffffffu, k2)) {
                abort_sh = 1;
              } else {
                tc_fence_after_sync();
                const uint32_t to = tO + (I % 3) * NC + lane_base;
#pragma unroll
                for (int h = 0; h < (CU + 15) / 16; ++h) {
                  float o[16];
                  tmem_ld16(to + 16 * h, o);
                  uint32_t ob[16];
#pragma unroll
                  for (int c = 0; c < 16; ++c)
                    ob[c] = __float_as_uint(16 * h + c < CU ? o[c] * alpha(16 * h + c) : o[c]);
                  tmem_st16_u(to + 16 * h, ob);
                }
                tmem_wait_st();
              }
            }
#pragma unroll
            for (int c = 0; c < CU; ++c) l_part[c] *= alpha(c);   // the sums follow
          }
#pragma unroll
          for (int c = 0; c < CU; ++c) mu_r[c] = mu_sh[nb_][c];
          ++nraise;
          fresh = false;
        }
        // P = 2^(x - reference) and the column sums; the row of P into shared memory
        // P alternates between two buffers: the product of tile J - 2 must have read this one
        const int pb = J & 1;
        bool k3 = J < 2 || waitb(pfree(pb), ((J >> 1) - 1) & 1);
        if (!__all_sync(0xffffffffu, k3)) abort_sh = 1;
        uint32_t pk[CU / 2];
#pragma unroll
        for (int c = 0; c < CU; c += 2) {
          // fmaxf drops the NaN of (-inf) - (-inf): a column without reference has no weight
          const float p0 = fast_exp2(fmaxf(x[c] - mu_r[c], -256.f));
          const float p1 = fast_exp2(fmaxf(x[c + 1] - mu_r[c + 1], -256.f));
          l_part[c] += p0;
          l_part[c + 1] += p1;
          pk[c / 2] = Mma<T>::pack(p0, p1);
        }
        const uint32_t prow = sP + pb * L::PBYTES + prow_off;
#pragma unroll
        for (int j = 0; j < CU / 8; ++j)
          asm volatile("st.shared.v4.b32 [%0], {%1,%2,%3,%4};" ::"r"(prow + ((j ^ pswz) << 4)), "r"(pk[4 * j]),
                       "r"(pk[4 * j + 1]), "r"(pk[4 * j + 2]), "r"(pk[4 * j + 3])
                       : "memory");
        // value rows past the last token (in its block) are stale: zero them
        if (jt == g.nt - 1) {
          const int last_blk = (g.ctx - 1) / kBlock;
          if (tok >= g.ctx && tok / kBlock == last_blk) {
            const int vs = J % kVStages;
            if (waitb(vfull(vs), (J / kVStages) & 1)) {
              const uint32_t vrow = sV + vs * kTileBytes;
#pragma unroll
              for (int h = 0; h < 2; ++h)
#pragma unroll
                for (int ch = 0; ch < 8; ++ch)
                  asm volatile("st.shared.v4.b32 [%0], {%1,%1,%1,%1};" ::"r"(vrow + h * kStrip + swz128(t, ch)),
                               "r"(0u)
                               : "memory");
            } else {
              abort_sh = 1;
            }
          }
        }
        fence_proxy_async_smem();
        tc_fence_before_sync();
        __syncwarp();
        if (lane == 0) mbar_arrive(pfull(pb));
        ++J;
      }
      if (stop) {
        ok = false;
        break;
      }
      // the segment's column sums and references for the epilogue
      const float lsum = warp_columns<CU, false>(l_part, lane);
      const int sbuf = I % 3;
      bool k4 = I < 3 || waiti(stfree(sbuf), ((I / 3) - 1) & 1);
      if (!__all_sync(0xffffffffu, k4)) abort_sh = 1;
      if (lane < CU) st_l[sbuf][warp][lane] = lsum;
      if (warp == 0 && lane < CU) st_m[sbuf][lane] = fresh ? -INFINITY : mu_sh[nraise & 1][lane];
      __syncwarp();
      if (lane == 0) mbar_arrive(stfull(sbuf));
      ++I;
    }
    if (!ok) abort_sh = 1;
  } else {
    // ---------------------------------------------------------- epilogue warps
    const int d = threadIdx.x - 128;                // head-dim row of O^T, TMEM lane d
    const uint32_t lane_base = static_cast<uint32_t>((warp & 3) * 32) << 16;
    // sequences with an empty context own no tile: their rows are zero
    for (int s = blockIdx.x; s < a.num_seqs; s += geff) {
      if (blockIdx.x >= geff) break;
      if (checked_context(a, s, false) != 0) continue;
      T* out = static_cast<T*>(a.out);
      for (int idx = d; idx < H * NQ * D; idx += 128) {
        const int kvh = idx / (NQ * D);
        const int rem = idx - kvh * NQ * D;
        out[query_row(a, s, kvh, G, rem / D) * D + rem % D] = Elem<T>::from_f(0.f);
      }
    }
    Walk w = make_walk();
    Segment g;
    int I = 0;
    bool ok = true;
    const int Hq = a.num_q_heads;
    while (next_segment(a, w, vtot, geff, g, ctx_sh, walk_i[0])) {
      const int ob = I % 3;
      bool k = waiti(ofull(ob), (I / 3) & 1);
      k = __all_sync(0xffffffffu, k) && waiti(stfull(ob), (I / 3) & 1);
      k = __all_sync(0xffffffffu, k);
      if (cta_any(2, !k)) {
        ok = false;
        break;
      }
      tc_fence_after_sync();
      float o[CU];
      load_cols<CU>(tO + ob * NC + lane_base, o);
      tc_fence_before_sync();
      // this thread's normalised output of every column; the statistics are copied out
      // so both buffers return to their producers at once
      float my_lse = -INFINITY;   // log2-sum-exp2 of column d (thread d stores it)
#pragma unroll
      for (int c = 0; c < CU; ++c) {
        const float l = (st_l[ob][0][c] + st_l[ob][1][c]) + (st_l[ob][2][c] + st_l[ob][3][c]);
        o[c] *= l > 0.f ? __frcp_rn(l) : 0.f;
        if (c == d && l > 0.f) my_lse = st_m[ob][c] + log2f(l);
      }
      __syncwarp();
      if (lane == 0) {
        mbar_arrive(ofree(ob));
        mbar_arrive(stfree(ob));
      }
      // output row of column c = i G + h: (s q_len + i) Hq + kvh G + h, walked without division
      const size_t row0 = static_cast<size_t>(g.s) * a.q_len * Hq + static_cast<size_t>(g.kvh) * G;
      if (g.n_parts == 1) {
        T* out = static_cast<T*>(a.out);
        size_t row = row0;
        int h = 0;
#pragma unroll
        for (int c = 0; c < CU; ++c) {
          if (c < NQ) out[row * D + d] = Elem<T>::from_f(o[c]);
          if (++h == G) {
            h = 0;
            row += Hq - G + 1;
          } else {
            ++row;
          }
        }
      } else {
        const int ms = a.max_splits;
        {
          size_t row = row0;
          int h = 0;
#pragma unroll
          for (int c = 0; c < CU; ++c) {
            if (c < NQ) {
              const size_t r = row * ms + g.part;
              a.ws_o[r * D + d] = o[c];
              if (d == c) a.ws_lse[r] = my_lse;
            }
            if (++h == G) {
              h = 0;
              row += Hq - G + 1;
            } else {
              ++row;
            }
          }
        }
        // the CTA that stores the last segment of (s, kvh) merges them all
        group_sync(2);
        int* counter = a.ws_count + static_cast<size_t>(g.s) * H + g.kvh;
        if (d == 0) {
          int prev;
          asm volatile("atom.add.acq_rel.gpu.global.s32 %0, [%1], 1;" : "=r"(prev) : "l"(counter) : "memory");
          last_sh = prev == g.n_parts - 1;
        }
        group_sync(2);
        if (last_sh) {
          // log-sum-exp over the partials, 8 columns at a time, one partial at a time with
          // a running maximum; each pass issues its 16 loads together
          T* out = static_cast<T*>(a.out);
#pragma unroll
          for (int cg = 0; cg < CU; cg += 8) {
            size_t rows[8];
            float M[8], Ls[8], Os[8];
#pragma unroll
            for (int k = 0; k < 8; ++k) {
              const int c = cg + k;
              rows[k] = query_row(a, g.s, g.kvh, G, c < NQ ? c : 0);
              M[k] = -INFINITY;
              Ls[k] = 0.f;
              Os[k] = 0.f;
            }
            for (int pp = 0; pp < g.n_parts; ++pp) {
              float lp[8], op[8];
#pragma unroll
              for (int k = 0; k < 8; ++k) {
                const size_t r = rows[k] * ms + pp;
                lp[k] = cg + k < NQ ? __ldcg(a.ws_lse + r) : -INFINITY;
                op[k] = cg + k < NQ ? __ldcg(a.ws_o + r * D + d) : 0.f;
              }
#pragma unroll
              for (int k = 0; k < 8; ++k) {
                if (lp[k] == -INFINITY) continue;   // an empty partial weighs nothing
                const float mn = fmaxf(M[k], lp[k]);
                const float r0 = fast_exp2(M[k] - mn);  // 0 while M is still -inf
                const float wgt = fast_exp2(lp[k] - mn);
                Ls[k] = Ls[k] * r0 + wgt;
                Os[k] = Os[k] * r0 + wgt * op[k];
                M[k] = mn;
              }
            }
#pragma unroll
            for (int k = 0; k < 8; ++k)
              if (cg + k < NQ) out[rows[k] * D + d] = Elem<T>::from_f(Ls[k] > 0.f ? Os[k] * __frcp_rn(Ls[k]) : 0.f);
          }
          if (d == 0) *counter = 0;   // zero again for the next call on this workspace
        }
        group_sync(2);
      }
      ++I;
    }
    if (!ok) abort_sh = 1;
  }

  // ------------------------------------------------------------------ teardown
  tc_fence_before_sync();
  __syncthreads();
  if (threadIdx.x == 0 && abort_sh) flag_status(a.status, PA_DEV_WAIT_TIMEOUT);
  if (warp == 0) {
    tc_fence_after_sync();
    tmem_dealloc(tmem, L::TMEM_COLS);
  }
}

namespace {

int sm_count() {
  static int n = [] {
    int dev = 0, v = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || cudaDeviceGetAttribute(&v, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess)
      return 0;
    return v;
  }();
  return n;
}

template <typename T, int CU>
cudaError_t launch_vu_t(const DecodeArgs& a, const CUtensorMap& kmap, const CUtensorMap& vmap, cudaStream_t stream) {
  constexpr int NC = CU <= 16 ? 16 : 32;
  const int smem = VLayout<NC>::SMEM + 1024;
  auto kern = verify_umma_kernel<T, NC, CU>;
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
  if (e != cudaSuccess) return e;
  const int sms = sm_count();
  if (sms <= 0) return cudaErrorNoDevice;
  return launch_pdl(kern, dim3(static_cast<unsigned>(sms)), dim3(kUThreads), smem, stream, kmap, vmap, a);
}

}  // namespace

int verify_umma_slots(int max_context_len, int part_blocks) {
  const int lmin = part_blocks >= kTileBlocks ? part_blocks / kTileBlocks : 1;
  const int nt = (max_context_len + kTok - 1) / kTok;
  return (nt + lmin - 1) / lmin + 2;
}

cudaError_t launch_verify_umma(const DecodeArgs& a, int dtype, const CUtensorMap& kmap, const CUtensorMap& vmap,
                               cudaStream_t stream) {
  // the softmax works on the used columns rounded up to 8 (one 16-byte chunk of a row of P)
  const int nq = (a.num_q_heads / a.num_kv_heads) * a.q_len;
  if (dtype == PA_BF16)
    return nq <= 8    ? launch_vu_t<__nv_bfloat16, 8>(a, kmap, vmap, stream)
           : nq <= 16 ? launch_vu_t<__nv_bfloat16, 16>(a, kmap, vmap, stream)
           : nq <= 24 ? launch_vu_t<__nv_bfloat16, 24>(a, kmap, vmap, stream)
                      : launch_vu_t<__nv_bfloat16, 32>(a, kmap, vmap, stream);
  return nq <= 8    ? launch_vu_t<__half, 8>(a, kmap, vmap, stream)
         : nq <= 16 ? launch_vu_t<__half, 16>(a, kmap, vmap, stream)
         : nq <= 24 ? launch_vu_t<__half, 24>(a, kmap, vmap, stream)
                    : launch_vu_t<__half, 32>(a, kmap, vmap, stream);
}

}  // namespace pa
