// pa_internal.h -- launch interface between the C ABI layer and the kernels.
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "pa.h"

namespace pa {

// Everything a decode launch needs; passed to the kernels by value.
struct DecodeArgs {
  void* out;
  const void* q;
  const void* k_pool;
  const void* v_pool;
  const int32_t* block_tables;
  const int32_t* context_lens;
  float scale_log2;        // softmax scale * log2(e): scores live in the log2 domain
  int num_seqs;
  int num_q_heads;
  int num_kv_heads;
  int head_dim;
  int max_blocks_per_seq;
  int max_context_len;     // host-known bound; larger device values are clamped
  int num_blocks;
  int part_blocks;         // pool blocks per split-K partition
  int max_splits;          // ceil(ceil(max_context_len / 16) / part_blocks)
  float* ws_o;             // [S][H_q][max_splits][D]  normalised partial outputs
  float* ws_lse;           // [S][H_q][max_splits]     partial log2-sum-exp2
  int* ws_count;           // [S][H_kv] partitions finished (zero between calls)
  int* status;             // device status word (PA_DEV_* bits)
  const float* k_scales;   // INT8 cache only: [N_blk][H_kv][16] row scales
  const float* v_scales;
  int q_len;               // query positions per sequence: 1 for decode, K+1 to verify K drafts
  // decode step with the append fused in: the new token of each sequence
  // ([S][H_kv][D] rows, written at position context - 1); null otherwise
  const void* k_new;
  const void* v_new;
};

struct PrefillArgs {
  void* out;
  const void* q;
  const int32_t* block_tables;
  const int32_t* cu_q_lens;
  const int32_t* context_lens;
  float scale_log2;
  int num_seqs;
  int num_q_heads;
  int num_kv_heads;
  int head_dim;
  int max_blocks_per_seq;
  int num_blocks;
  int max_q_len;
  int* status;
  int* sched;   // the launch's pair of schedule counters (items taken, CTAs finished), zero on entry
};

// Record `msg` as the calling thread's pa_last_error() and return `code`.
int set_last_error(int code, const char* msg);

// The calling thread's current CUDA context (driver handle), or null.  Device
// addresses of the library's __device__ variables are cached per (device,
// context): a device reset creates a new context, whose module may place them
// elsewhere, so a changed handle triggers a fresh lookup.
void* current_context();

// Streaming multiprocessors of the current device (queried once per device;
// 0 when no device is current).
int device_sm_count();

cudaError_t launch_append(void* k_pool, void* v_pool, const int64_t* slot_mapping,
                          const void* k_new, const void* v_new, int num_tokens,
                          int num_kv_heads, int row_bytes, int num_blocks, int* status,
                          cudaStream_t stream);

// Tensor-core decode (bf16/fp16 pools, D in {64, 128}, G <= 8).
cudaError_t launch_decode_tc(const DecodeArgs& a, int dtype, const CUtensorMap& kmap,
                             const CUtensorMap& vmap, cudaStream_t stream);

// Verification attention (q_len > 1 query positions per sequence, bf16/fp16):
// one consumer warp per 8 query columns over a CTA-shared ring of K/V stages.
cudaError_t launch_verify_tc(const DecodeArgs& a, int dtype, const CUtensorMap& kmap,
                             const CUtensorMap& vmap, cudaStream_t stream);

// Verification attention on the tensor cores (tcgen05), head dim 128, q_len > 1:
// a persistent stream-K launch, one CTA per SM.  a.part_blocks / 8 is the
// shortest range of 128-token tiles a CTA takes; a.max_splits must be
// verify_umma_slots(max_context_len, part_blocks) (partials per output row).
cudaError_t launch_verify_umma(const DecodeArgs& a, int dtype, const CUtensorMap& kmap,
                               const CUtensorMap& vmap, cudaStream_t stream);
int verify_umma_slots(int max_context_len, int part_blocks);

// CUDA-core decode (any supported dtype; the fp32 path).
cudaError_t launch_decode_simt(const DecodeArgs& a, int dtype, cudaStream_t stream);

// INT8 cache: quantise-on-append of bf16/fp16 rows (act_dtype), and decode
// over int8 codes with float32 row scales (q / out in act_dtype).
cudaError_t launch_append_q8(void* k_codes, void* v_codes, float* k_scales, float* v_scales,
                             const int64_t* slot_mapping, const void* k_new, const void* v_new, int num_tokens,
                             int num_kv_heads, int head_dim, int act_dtype, int num_blocks, int* status,
                             cudaStream_t stream);
cudaError_t launch_decode_q8(const DecodeArgs& a, int act_dtype, const CUtensorMap& kmap,
                             const CUtensorMap& vmap, cudaStream_t stream);

// Rotary position embedding: the (cos, sin) table, K rotated on append, rows in place.
cudaError_t launch_rope_cache(float* cos_sin, int max_positions, int head_dim, double theta, cudaStream_t stream);
cudaError_t launch_append_rope(void* k_pool, void* v_pool, const int64_t* slot_mapping, const int32_t* positions,
                               const void* k_new, const void* v_new, const float* cos_sin, int max_positions,
                               int num_tokens, int num_kv_heads, int head_dim, int dtype, int num_blocks,
                               int* status, cudaStream_t stream);
cudaError_t launch_apply_rope(void* x, const int32_t* positions, const float* cos_sin, int max_positions,
                              int num_tokens, int num_heads, int head_dim, int dtype, int* status,
                              cudaStream_t stream);

// Copy-on-write: whole blocks of up to four block-indexed arrays (K and V
// pools; for an INT8 cache also the K and V scale arrays), pairs (src, dst)
// on the device.  chunks_per_block = 16-byte chunks of one block in that array.
struct CopyArrays {
  void* ptr[4];
  int chunks_per_block[4];
};
cudaError_t launch_copy_blocks(const CopyArrays& arrs, int num_arrays, const int32_t* pairs, int num_pairs,
                               int num_blocks, int* status, cudaStream_t stream);

// The blocks of each sequence's first context_lens[s] positions of an INT8
// cache, dequantised to fp16 into a pool of num_seqs * B blocks (k_out,
// v_out), sequence s owning blocks s * B .. s * B + B - 1, with the block
// table table_out[s][lb] = s * B + lb.  A block id outside the pool sets
// PA_DEV_BAD_BLOCK_ID and gives zeros; a value past fp16's range is clamped
// and sets PA_DEV_RANGE.
struct DequantQ8Args {
  const int8_t* k_codes;
  const int8_t* v_codes;
  const float* k_scales;
  const float* v_scales;
  const int32_t* block_tables;
  const int32_t* context_lens;
  int num_seqs, max_blocks_per_seq, num_kv_heads, head_dim, num_blocks, B;
  void* k_out;   // fp16
  void* v_out;   // fp16
  int32_t* table_out;
  int* status;
};
cudaError_t launch_dequant_q8(const DequantQ8Args& a, cudaStream_t stream);

// Causal prefill on tcgen05 with tensor-memory accumulators (bf16/fp16, D in {64, 128}).
// dtype: the pools and the products; act_dtype: q and the output rows (dtype,
// or PA_BF16 over an fp16 pool: the pass converts q in shared memory).
// qmap: the queries as (D, H, rows) in 128-row x 64-column boxes (whole query tiles only).
cudaError_t launch_prefill_umma(const PrefillArgs& a, int dtype, int act_dtype, const CUtensorMap& kmap,
                                const CUtensorMap& vmap, const CUtensorMap& qmap, cudaStream_t stream);


}  // namespace pa
