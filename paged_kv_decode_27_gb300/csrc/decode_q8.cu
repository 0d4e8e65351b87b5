// decode_q8.cu -- paged decode attention over an INT8 KV cache, and the
// verification pass of speculative decoding over the same cache.
//
// The cache holds K and V quantised per token head ("LLM Inference Server",
// Optional Bonus Extensions: INT8 KV-Cache Quantization; rule of its Required
// Mathematical Concepts: x_hat = s * x_q): int8 codes in the float pool's
// layout plus one float32 scale per (block, head, slot).  Decode reads half
// the bytes of a bf16 cache and stays bound by HBM bandwidth, so the work
// split is that of the bf16 kernel -- grid (split, KV head, sequence), one
// CTA per partition with all G query heads of the group, four warps each
// running its own TMA pipeline -- and the codes are widened in registers:
//
//  * Codes to fp16 without a conversion unit: a code byte XOR 0x80 is
//    code + 128 as an unsigned byte u, and the fp16 bit pattern 0x64uu is
//    1024 + u, i.e. 1152 + code exactly.  One byte permute builds two such
//    halves.  The offset stays in the MMA operands and is removed from the
//    fp32 results: from the scores by subtracting 1152 * sum_d q[d] (computed
//    once per CTA with the same MMA on a constant operand), from the output by
//    a ninth MMA per block on the constant that accumulates 1152 * sum_i p_i
//    alongside O.  The offset is ~9x the largest code, so it adds ~9x the
//    fp32 accumulation error to a score: about 1e-5 of the score's size.
//  * Scores, S^T = K q^T with mma.sync m16n8k16 in fp16: tokens are M, the
//    query group (padded to 8) is N.  q is brought into fp16 exactly by a
//    power-of-two row scale 2^e (its largest element lands in [2^14, 2^15)),
//    folded back into the softmax scale.  The head dimension is visited in a
//    permuted order -- k-slots (2c, 2c+1, 2c+8, 2c+9) of k-step j hold
//    d = 16c + 4j + (0, 1, 2, 3) -- so that a lane's A fragments for one token
//    row come from one 16-byte shared-memory load; q uses the same order.
//    Score = (S - 1152 sum q) * scale * log2(e) * 2^-e * s_k[token].
//  * MMA row m holds token tau(m) = m ^ ((m & 1) << 2): with the 128-byte
//    swizzle this keeps both the K-row loads (rows g, g+8) and the V-row loads
//    (tokens of k-slots 2c.., one per quad) free of bank conflicts.
//  * Output, O^T = V^T P^T: a lane's A fragments cover a contiguous run of
//    D/8 head-dim entries of each of its 4 tokens (one load per token); m-tile
//    j row g is d = (D/8) g + 2j and row g+8 is d + 1.  P^T (the B operand,
//    from the score accumulators by movmatrix) carries p_i * s_v[i] / M where
//    M is the running maximum of s_v over the warp's tokens, so it stays in
//    [0, 1] whatever the value range; when M grows the accumulators are
//    rescaled with the softmax's own correction, and the warp's O is
//    multiplied by M at the end.  Positions past the context have p = 0 (their
//    codes are finite integers and their scales are never read into p).
//
// Verification ("LLM Inference Server", Batched Scheduling & Speculative
// Decoding: q_len = K + 1 query tokens per sequence) widens N: the q_len x G
// query columns of a KV head fill NT 8-column tiles that share every widened
// K and V fragment, and key j is masked from query i unless
// j <= ctx - q_len + i.  Each tile holds its own accumulators, so NT > 1 runs
// 2 CTAs per SM.
//
// The warps' states merge in shared memory and the split-K partials by
// log-sum-exp exactly as in the float kernels (decode_merge.cuh).
#include "decode_merge.cuh"
#include "pa_common.cuh"
#include "pa_internal.h"

namespace pa {

namespace {

constexpr uint32_t kMagic = 0x64646464u;    // fp16 exponent byte of 1024 + u
constexpr uint32_t kBiasPair = 0x64806480u; // fp16 (1152, 1152)
constexpr uint32_t kFlip = 0x80808080u;     // int8 code -> code + 128 as u8
constexpr float kLazy = 8.f;                // log2 headroom of the softmax reference

__device__ __forceinline__ int tau(int m) { return m ^ ((m & 1) << 2); }

// bytes b0, b1 (sel 0x4140) or b2, b3 (sel 0x4342) of w as two fp16 1024 + b
__device__ __forceinline__ uint32_t widen(uint32_t w, uint32_t sel) { return __byte_perm(w, kMagic, sel); }

__device__ __forceinline__ uint32_t pack_half2(float lo, float hi) {
  __half2 v = __floats2half2_rn(lo, hi);
  return *reinterpret_cast<uint32_t*>(&v);
}

__device__ __forceinline__ uint2 lds64(uint32_t addr) {
  uint2 v;
  asm volatile("ld.shared.v2.u32 {%0,%1}, [%2];" : "=r"(v.x), "=r"(v.y) : "r"(addr));
  return v;
}

// Byte offset of the 16-byte chunk `ch` of code row `r` inside a tile (rows of
// D bytes; 128-byte swizzle for D = 128, 64-byte swizzle for D = 64).
template <int D>
__device__ __forceinline__ uint32_t tile_chunk(int r, int ch) {
  if (D == 128) return static_cast<uint32_t>(r * 128 + ((ch ^ (r & 7)) << 4));
  return static_cast<uint32_t>(r * 64 + ((ch ^ ((r >> 1) & 3)) << 4));
}

// A lane's D/8-byte run of row r starting at head-dim entry (D/8) * g.
template <int D> struct VRun;
template <> struct VRun<128> {
  static constexpr int WORDS = 4;
  static __device__ __forceinline__ void load(uint32_t tile, int r, int g, uint32_t* w) {
    const uint4 v = lds128(tile + tile_chunk<128>(r, g));
    w[0] = v.x ^ kFlip; w[1] = v.y ^ kFlip; w[2] = v.z ^ kFlip; w[3] = v.w ^ kFlip;
  }
};
template <> struct VRun<64> {
  static constexpr int WORDS = 2;
  static __device__ __forceinline__ void load(uint32_t tile, int r, int g, uint32_t* w) {
    const uint2 v = lds64(tile + tile_chunk<64>(r, g >> 1) + ((g & 1) << 3));
    w[0] = v.x ^ kFlip; w[1] = v.y ^ kFlip;
  }
};

}  // namespace

// NT 8-column tiles of query columns (column c = i * G + h for query position
// i and head h, as in decode_merge.cuh); CAUSAL masks key j from query i
// unless j <= ctx - q_len + i.  Decode is NT = 1 without the mask.
template <typename T, int D, int W, int NS, int NT, bool CAUSAL>
__global__ void __launch_bounds__(W * 32, NT == 1 ? 4 : 2)
decode_q8_kernel(const __grid_constant__ CUtensorMap kmap, const __grid_constant__ CUtensorMap vmap,
                 const DecodeArgs a) {
  constexpr int TILE = 16 * D;         // one (block, head) tile of codes
  constexpr int STAGE = 2 * TILE;      // K tile then V tile
  constexpr int KS = D / 16;           // k-steps of the score MMA = m-tiles of the PV MMA
  constexpr int HALVES = D / 64;       // 64-entry halves of the head dim
  constexpr int RUNW = VRun<D>::WORDS; // words of a lane's V run
  constexpr int NC = 8 * NT;           // query columns per warp state

  extern __shared__ uint8_t smem_raw[];
  __shared__ __align__(8) uint64_t bars[W * NS];
  __shared__ __align__(16) float scl[W * NS][2][kBlock];   // per stage: K scales, V scales
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                             ~static_cast<uintptr_t>(1023));

  const int split = blockIdx.x;
  const int kvh = blockIdx.y;
  const int s = blockIdx.z;
  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const int G = a.num_q_heads / a.num_kv_heads;
  const int ncols = CAUSAL ? G * a.q_len : G;

  grid_dependency_wait();   // the codes may come from the append just before us
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
  const uint32_t sbase = smem_u32(&scl[warp * NS][0][0]);
  const uint32_t bar0 = smem_u32(&bars[warp * NS]);
  const uint64_t policy = l2_policy_evict_first();
  if (lane == 0) {
    for (int st = 0; st < NS; ++st) mbar_init(bar0 + 8 * st, 1);
    fence_barrier_init();
    prefetch_tensormap(&kmap);
    prefetch_tensormap(&vmap);
  }
  __syncwarp();

  auto issue = [&](int i) {
    const int id = __shfl_sync(0xffffffffu, my_id, i);
    if (lane == 0) {
      const int st = i % NS;
      const uint32_t bar = bar0 + 8 * st;
      const uint32_t dst = wbase + st * STAGE;
      const int y = (id * a.num_kv_heads + kvh) * kBlock;
      const size_t srow = static_cast<size_t>(id * a.num_kv_heads + kvh) * kBlock;
      mbar_arrive_expect_tx(bar, STAGE + 2 * kBlock * 4);
      tma_load_2d(dst, &kmap, 0, y, bar, policy);
      tma_load_2d(dst + TILE, &vmap, 0, y, bar, policy);
      bulk_load(sbase + st * 2 * kBlock * 4, a.k_scales + srow, kBlock * 4, bar);
      bulk_load(sbase + st * 2 * kBlock * 4 + kBlock * 4, a.v_scales + srow, kBlock * 4, bar);
    }
  };
  const int npro = nb_w < NS ? nb_w : NS;
  for (int i = 0; i < npro; ++i) issue(i);

  const int g = lane >> 2;   // fragment row group
  const int c = lane & 3;    // thread in group

  // ---- q in fp16, exactly, with a power-of-two row scale ---------------------
  // B operand of the score MMA: k-step ks = 4 h + j of tile nt holds, for this
  // lane, q[column 8 nt + g][64 h + 16 c + 4 j + (0, 1)] and (+2, +3).
  uint32_t qf[NT][KS][2];
  float f0[NT], f1[NT];   // scale * log2(e) * 2^-e of this lane's score columns 2c, 2c+1
#pragma unroll
  for (int nt = 0; nt < NT; ++nt) {
    const int col = 8 * nt + g;
    float qv[HALVES * 16];
    if (col < ncols) {
      const int qi = col / G;
      const int h = col - qi * G;
      const T* qrow = static_cast<const T*>(a.q) +
                      ((static_cast<size_t>(s) * a.q_len + qi) * a.num_q_heads + kvh * G + h) * D;
#pragma unroll
      for (int hf = 0; hf < HALVES; ++hf) {
        const uint4* p = reinterpret_cast<const uint4*>(qrow + 64 * hf + 16 * c);
        const uint4 u0 = __ldg(p), u1 = __ldg(p + 1);
        const T* e0 = reinterpret_cast<const T*>(&u0);
        const T* e1 = reinterpret_cast<const T*>(&u1);
#pragma unroll
        for (int i = 0; i < 8; ++i) {
          qv[hf * 16 + i] = Elem<T>::to_f(e0[i]);
          qv[hf * 16 + 8 + i] = Elem<T>::to_f(e1[i]);
        }
      }
    } else {
#pragma unroll
      for (int i = 0; i < HALVES * 16; ++i) qv[i] = 0.f;
    }
    float amax = 0.f;
#pragma unroll
    for (int i = 0; i < HALVES * 16; ++i) amax = fmaxf(amax, fabsf(qv[i]));
    amax = warp_max_xor(amax, 1, 2);
    int e = 0;
    if (amax > 0.f) {
      e = 141 - static_cast<int>((__float_as_uint(amax) >> 23) & 0xffu);   // amax * 2^e in [2^14, 2^15)
      e = e > 126 ? 126 : (e < -126 ? -126 : e);
    }
    const float up = __uint_as_float(static_cast<uint32_t>(e + 127) << 23);
    const float f_head = a.scale_log2 * __uint_as_float(static_cast<uint32_t>(127 - e) << 23);
#pragma unroll
    for (int hf = 0; hf < HALVES; ++hf) {
#pragma unroll
      for (int j = 0; j < 4; ++j) {
        const float* v = qv + hf * 16 + 4 * j;
        qf[nt][hf * 4 + j][0] = pack_half2(v[0] * up, v[1] * up);
        qf[nt][hf * 4 + j][1] = pack_half2(v[2] * up, v[3] * up);
      }
    }
    f0[nt] = __shfl_sync(0xffffffffu, f_head, 8 * c);
    f1[nt] = __shfl_sync(0xffffffffu, f_head, 8 * c + 4);
  }
  const uint32_t cbias[4] = {kBiasPair, kBiasPair, kBiasPair, kBiasPair};
  // 1152 * sum_d q16[column][d]: [0],[2] column 2c; [1],[3] column 2c+1 of each tile
  float bq[NT][4];
#pragma unroll
  for (int nt = 0; nt < NT; ++nt) {
    bq[nt][0] = bq[nt][1] = bq[nt][2] = bq[nt][3] = 0.f;
#pragma unroll
    for (int ks = 0; ks < KS; ++ks) Mma<__half>::run(bq[nt], cbias, qf[nt][ks][0], qf[nt][ks][1]);
  }
  // keys visible to this lane's score columns: ctx - q_len + 1 + i for query
  // position i, none for padding columns
  int lim[NT][2];
#pragma unroll
  for (int nt = 0; nt < NT; ++nt) {
#pragma unroll
    for (int u = 0; u < 2; ++u) {
      const int col = 8 * nt + 2 * c + u;
      lim[nt][u] = CAUSAL ? (col < ncols ? ctx - a.q_len + 1 + col / G : 0) : ctx;
    }
  }

  // Softmax state of this lane's columns in the log2 domain.  m_ref is a
  // lazily raised reference: it moves only when a score exceeds it by more
  // than kLazy, so unnormalised weights stay <= 2^kLazy and most blocks need
  // no reduction and no rescale.  sv_ref plays the same role for the V scales.
  float m_ref[NT][2], mu[NT][2], l_run[NT][2];   // mu: m_ref, or 0 while it is -inf
  float sv_ref = 0.f, sv_inv = 0.f;
  float acc[NT][KS][4];
  float bo[NT][4];   // 1152 * sum_i p''_i, accumulated like O
#pragma unroll
  for (int nt = 0; nt < NT; ++nt) {
    m_ref[nt][0] = m_ref[nt][1] = -INFINITY;
    mu[nt][0] = mu[nt][1] = 0.f;
    l_run[nt][0] = l_run[nt][1] = 0.f;
    bo[nt][0] = bo[nt][1] = bo[nt][2] = bo[nt][3] = 0.f;
#pragma unroll
    for (int mt = 0; mt < KS; ++mt) acc[nt][mt][0] = acc[nt][mt][1] = acc[nt][mt][2] = acc[nt][mt][3] = 0.f;
  }

  const int r0 = tau(g), r1 = tau(g + 8);                    // token rows of the score accumulators
  const int tx = tau(2 * c), ty = tau(2 * c + 1);            // tokens of PV k-slots 2c, 2c+1
  const int tz = tau(2 * c + 8), tw = tau(2 * c + 9);        //                     2c+8, 2c+9

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
    const float* sk = &scl[warp * NS + st][0][0];
    const float* sv = &scl[warp * NS + st][1][0];
    const int lb = blk0 + warp + i * W;
    int nvalid = ctx - lb * kBlock;
    nvalid = nvalid > kBlock ? kBlock : nvalid;
    if (bad_mask & (1u << i)) nvalid = 0;

    // ---- scores -----------------------------------------------------------
    float sa[NT][4], sb[NT][4];
#pragma unroll
    for (int nt = 0; nt < NT; ++nt) {
      sa[nt][0] = sa[nt][1] = sa[nt][2] = sa[nt][3] = 0.f;
      sb[nt][0] = sb[nt][1] = sb[nt][2] = sb[nt][3] = 0.f;
    }
#pragma unroll
    for (int hf = 0; hf < HALVES; ++hf) {
      uint4 A = lds128(kt + tile_chunk<D>(r0, 4 * hf + c));
      uint4 B = lds128(kt + tile_chunk<D>(r1, 4 * hf + c));
      const uint32_t wa[4] = {A.x ^ kFlip, A.y ^ kFlip, A.z ^ kFlip, A.w ^ kFlip};
      const uint32_t wb[4] = {B.x ^ kFlip, B.y ^ kFlip, B.z ^ kFlip, B.w ^ kFlip};
#pragma unroll
      for (int j = 0; j < 4; ++j) {
        const uint32_t af[4] = {widen(wa[j], 0x4140), widen(wb[j], 0x4140), widen(wa[j], 0x4342),
                                widen(wb[j], 0x4342)};
#pragma unroll
        for (int nt = 0; nt < NT; ++nt) {
          if (j & 1)
            Mma<__half>::run(sb[nt], af, qf[nt][hf * 4 + j][0], qf[nt][hf * 4 + j][1]);
          else
            Mma<__half>::run(sa[nt], af, qf[nt][hf * 4 + j][0], qf[nt][hf * 4 + j][1]);
        }
      }
    }
    const bool v0 = r0 < nvalid, v1 = r1 < nvalid;
    const float sk0 = v0 ? sk[r0] : 0.f;
    const float sk1 = v1 ? sk[r1] : 0.f;
    const float sv0 = v0 ? sv[r0] : 0.f;
    const float sv1 = v1 ? sv[r1] : 0.f;
    float x[NT][4];
#pragma unroll
    for (int nt = 0; nt < NT; ++nt) {
      bool m0 = v0, m1 = v0, m2 = v1, m3 = v1;   // (token r0 | r1) x (column 2c | 2c+1)
      if (CAUSAL) {
        const int base = lb * kBlock;
        m0 = v0 && r0 < lim[nt][0] - base;
        m1 = v0 && r0 < lim[nt][1] - base;
        m2 = v1 && r1 < lim[nt][0] - base;
        m3 = v1 && r1 < lim[nt][1] - base;
      }
      x[nt][0] = m0 ? (sa[nt][0] + sb[nt][0] - bq[nt][0]) * (f0[nt] * sk0) : -INFINITY;
      x[nt][1] = m1 ? (sa[nt][1] + sb[nt][1] - bq[nt][1]) * (f1[nt] * sk0) : -INFINITY;
      x[nt][2] = m2 ? (sa[nt][2] + sb[nt][2] - bq[nt][2]) * (f0[nt] * sk1) : -INFINITY;
      x[nt][3] = m3 ? (sa[nt][3] + sb[nt][3] - bq[nt][3]) * (f1[nt] * sk1) : -INFINITY;
    }

    // ---- raise the references (rare) -----------------------------------------
    bool grow = fmaxf(sv0, sv1) > sv_ref;
#pragma unroll
    for (int nt = 0; nt < NT; ++nt)
      grow = grow || fmaxf(x[nt][0], x[nt][2]) > m_ref[nt][0] + kLazy ||
             fmaxf(x[nt][1], x[nt][3]) > m_ref[nt][1] + kLazy;
    if (__any_sync(0xffffffffu, grow)) {
      const float svb = warp_max_xor(fmaxf(sv0, sv1), 4, 16);
      const float svn = svb > sv_ref ? 2.f * svb : sv_ref;   // headroom: fewer raises
      const float rs = svn > 0.f ? sv_ref / svn : 1.f;
#pragma unroll
      for (int nt = 0; nt < NT; ++nt) {
        const float mb0 = warp_max_xor(fmaxf(x[nt][0], x[nt][2]), 4, 16);
        const float mb1 = warp_max_xor(fmaxf(x[nt][1], x[nt][3]), 4, 16);
        const float mn0 = fmaxf(m_ref[nt][0], mb0);
        const float mn1 = fmaxf(m_ref[nt][1], mb1);
        const float al0 = fast_exp2(m_ref[nt][0] - (mn0 == -INFINITY ? 0.f : mn0));
        const float al1 = fast_exp2(m_ref[nt][1] - (mn1 == -INFINITY ? 0.f : mn1));
        l_run[nt][0] *= al0;
        l_run[nt][1] *= al1;
        const float be0 = al0 * rs, be1 = al1 * rs;
#pragma unroll
        for (int mt = 0; mt < KS; ++mt) {
          acc[nt][mt][0] *= be0;
          acc[nt][mt][1] *= be1;
          acc[nt][mt][2] *= be0;
          acc[nt][mt][3] *= be1;
        }
        bo[nt][0] *= be0;
        bo[nt][1] *= be1;
        bo[nt][2] *= be0;
        bo[nt][3] *= be1;
        m_ref[nt][0] = mn0;
        m_ref[nt][1] = mn1;
        mu[nt][0] = mn0 == -INFINITY ? 0.f : mn0;
        mu[nt][1] = mn1 == -INFINITY ? 0.f : mn1;
      }
      sv_ref = svn;
      sv_inv = svn > 0.f ? __frcp_rn(svn) : 0.f;
    }
    const float w0 = sv0 * sv_inv, w1 = sv1 * sv_inv;   // s_v / sv_ref in [0, 1/2]
    uint32_t pb0[NT], pb1[NT];
#pragma unroll
    for (int nt = 0; nt < NT; ++nt) {
      const float p0 = fast_exp2(x[nt][0] - mu[nt][0]);
      const float p1 = fast_exp2(x[nt][1] - mu[nt][1]);
      const float p2 = fast_exp2(x[nt][2] - mu[nt][0]);
      const float p3 = fast_exp2(x[nt][3] - mu[nt][1]);
      l_run[nt][0] += p0 + p2;
      l_run[nt][1] += p1 + p3;
      pb0[nt] = movmatrix_trans(pack_half2(p0 * w0, p1 * w0));
      pb1[nt] = movmatrix_trans(pack_half2(p2 * w1, p3 * w1));
    }

    // ---- O^T[d][column] += V^T[d][token] P^T[token][column] ------------------
    uint32_t X[RUNW], Y[RUNW], Z[RUNW], Wr[RUNW];
    VRun<D>::load(vt, tx, g, X);
    VRun<D>::load(vt, ty, g, Y);
    VRun<D>::load(vt, tz, g, Z);
    VRun<D>::load(vt, tw, g, Wr);
#pragma unroll
    for (int mt = 0; mt < KS; ++mt) {
      const uint32_t sel = (mt & 1) ? 0x7362u : 0x5140u;
      const uint32_t t0 = __byte_perm(X[mt >> 1], Y[mt >> 1], sel);
      const uint32_t t1 = __byte_perm(Z[mt >> 1], Wr[mt >> 1], sel);
      const uint32_t vf[4] = {widen(t0, 0x4140), widen(t0, 0x4342), widen(t1, 0x4140), widen(t1, 0x4342)};
#pragma unroll
      for (int nt = 0; nt < NT; ++nt) Mma<__half>::run(acc[nt][mt], vf, pb0[nt], pb1[nt]);
    }
#pragma unroll
    for (int nt = 0; nt < NT; ++nt) Mma<__half>::run(bo[nt], cbias, pb0[nt], pb1[nt]);

    __syncwarp();
    if (i + NS < nb_w) {
      fence_proxy_async_smem();
      issue(i + NS);
    }
  }

  if (!ok) {
    if (lane == 0) flag_status(a.status, PA_DEV_WAIT_TIMEOUT);
    const int last = (i + NS < nb_w) ? i + NS : nb_w;
    for (int j = i; j < last; ++j) mbar_wait_bounded(bar0 + 8 * (j % NS), (j / NS) & 1, 100000000ull);
  }

  // ---- merge the W warp states through shared memory -------------------------
  __syncthreads();
  float* red_o = reinterpret_cast<float*>(smem);
  float* red_m = red_o + W * NC * D;
  float* red_l = red_m + W * NC;
  constexpr int RUN = D / 8;
#pragma unroll
  for (int nt = 0; nt < NT; ++nt) {
    l_run[nt][0] = warp_sum_xor(l_run[nt][0], 4, 16);
    l_run[nt][1] = warp_sum_xor(l_run[nt][1], 4, 16);
    const int h0 = 8 * nt + 2 * c;
    const int h1 = h0 + 1;
#pragma unroll
    for (int mt = 0; mt < KS; ++mt) {
      const int d0 = RUN * g + 2 * mt;
      if (h0 < ncols) {
        red_o[(warp * NC + h0) * D + d0] = (acc[nt][mt][0] - bo[nt][0]) * sv_ref;
        red_o[(warp * NC + h0) * D + d0 + 1] = (acc[nt][mt][2] - bo[nt][2]) * sv_ref;
      }
      if (h1 < ncols) {
        red_o[(warp * NC + h1) * D + d0] = (acc[nt][mt][1] - bo[nt][1]) * sv_ref;
        red_o[(warp * NC + h1) * D + d0 + 1] = (acc[nt][mt][3] - bo[nt][3]) * sv_ref;
      }
    }
    if (g == 0) {
      if (h0 < ncols) {
        red_m[warp * NC + h0] = m_ref[nt][0];
        red_l[warp * NC + h0] = l_run[nt][0];
      }
      if (h1 < ncols) {
        red_m[warp * NC + h1] = m_ref[nt][1];
        red_l[warp * NC + h1] = l_run[nt][1];
      }
    }
  }
  __syncthreads();
  cta_merge_store<T, W, D, NC>(a, red_o, red_m, red_l, G, s, kvh, split, n_splits);
}

namespace {

template <typename T, int D, int NT, bool CAUSAL>
cudaError_t launch_q8_t(const DecodeArgs& a, const CUtensorMap& kmap, const CUtensorMap& vmap,
                        cudaStream_t stream) {
  constexpr int W = 4;
  // Decode: 48 KB of stages per CTA, 4 CTAs (16 warps) per SM.  The loop is
  // bound by instruction issue, so more warps per SM beat deeper per-warp
  // pipelines (the same bytes in flight with 4 stages and 3 CTAs ran ~9%
  // slower).  Wider query tiles hold more accumulators per thread and run 2
  // CTAs per SM with one more stage each.
  constexpr int NS = NT == 1 ? ((D == 128) ? 3 : 6) : ((D == 128) ? 4 : 8);
  constexpr int STAGE = 2 * 16 * D;
  constexpr int NC = 8 * NT;
  constexpr int MERGE = W * NC * D * 4 + 2 * W * NC * 4;
  constexpr int BODY = W * NS * STAGE > MERGE ? W * NS * STAGE : MERGE;
  const int smem = BODY + 1024;
  auto kern = decode_q8_kernel<T, D, W, NS, NT, CAUSAL>;
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
  if (e != cudaSuccess) return e;
  dim3 grid(a.max_splits, a.num_kv_heads, a.num_seqs);
  return launch_pdl(kern, grid, dim3(W * 32), smem, stream, kmap, vmap, a);
}

template <typename T, int D>
cudaError_t launch_q8_d(const DecodeArgs& a, const CUtensorMap& kmap, const CUtensorMap& vmap,
                        cudaStream_t stream) {
  if (a.q_len == 1) return launch_q8_t<T, D, 1, false>(a, kmap, vmap, stream);
  const int tiles = ((a.num_q_heads / a.num_kv_heads) * a.q_len + 7) / 8;   // <= 4 (host limit)
  switch (tiles) {
    case 1: return launch_q8_t<T, D, 1, true>(a, kmap, vmap, stream);
    case 2: return launch_q8_t<T, D, 2, true>(a, kmap, vmap, stream);
    case 3: return launch_q8_t<T, D, 3, true>(a, kmap, vmap, stream);
    default: return launch_q8_t<T, D, 4, true>(a, kmap, vmap, stream);
  }
}

}  // namespace

cudaError_t launch_decode_q8(const DecodeArgs& a, int act_dtype, const CUtensorMap& kmap,
                             const CUtensorMap& vmap, cudaStream_t stream) {
  if (act_dtype == PA_BF16) {
    return a.head_dim == 128 ? launch_q8_d<__nv_bfloat16, 128>(a, kmap, vmap, stream)
                             : launch_q8_d<__nv_bfloat16, 64>(a, kmap, vmap, stream);
  }
  return a.head_dim == 128 ? launch_q8_d<__half, 128>(a, kmap, vmap, stream)
                           : launch_q8_d<__half, 64>(a, kmap, vmap, stream);
}

}  // namespace pa
