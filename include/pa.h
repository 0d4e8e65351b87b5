/*
 * pa.h -- C ABI of libpa: paged KV-cache attention for GB300 (sm_103a).
 *
 * The library implements the attention slice of an LLM inference engine whose
 * KV cache is a pool of fixed 16-token blocks shared by all requests
 * ("Mini inference engine (KV cache + sampling + quantization)", step 2 and
 * its stretch goal; "LLM Inference Server", Optional Bonus Extensions:
 * Paged KV-Cache Block Allocator; "LLM Inference Server From Scratch",
 * How it works, 3 Block Manager and 4 Attention Kernel).
 *
 * Conventions shared by every call
 * --------------------------------
 *  - Every tensor pointer is a DEVICE pointer owned by the caller.  The library
 *    allocates no device memory, never synchronises, and enqueues its kernels
 *    on `stream` (a cudaStream_t passed as void*; NULL = the legacy default
 *    stream).  Results are ready when the stream reaches that point.
 *  - Pool layout, identical for K and V: [num_blocks][num_kv_heads][16][head_dim],
 *    row-major, element type `dtype`.  Each (block, head) tile is one contiguous
 *    16*head_dim*elem_bytes run.  Token position p of a sequence lives in
 *    logical block p/16 at offset p%16; logical block j is physical block
 *    block_tables[seq*max_blocks_per_seq + j].
 *  - Grouped-query attention: q head h reads KV head h / (num_q_heads/num_kv_heads).
 *  - context_lens[s] counts every cached token of sequence s, including the
 *    token appended in this step (the new token is at position context_len-1).
 *  - q, K, V and out share one dtype; scores, softmax and accumulation run in
 *    fp32; out is rounded to the dtype once (round-to-nearest-even).
 *  - Return value: PA_OK, or a negative code with a message in pa_last_error().
 *    All argument checks run on the host BEFORE anything is enqueued, so a
 *    rejected call leaves the stream and the device untouched.  Device-side
 *    data (slots, block ids, context lengths) is range-checked in the kernels:
 *    an out-of-range value is skipped and recorded in a device status word
 *    (see pa_device_status), never dereferenced.
 */
#ifndef PA_H_
#define PA_H_

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

#if defined(__GNUC__)
#define PA_API __attribute__((visibility("default")))
#else
#define PA_API
#endif

#define PA_BLOCK_SIZE 16
#define PA_VERSION 1

/* PA_I8 is the element type of an INT8 KV cache only (pools of int8 codes with
 * a float32 scale per row, see pa_append_kv_int8); q, out and new K/V rows are
 * never int8. */
typedef enum { PA_F32 = 0, PA_BF16 = 1, PA_F16 = 2, PA_I8 = 3 } pa_dtype;

enum {
  PA_OK = 0,
  PA_ERR_INVALID = -1,     /* bad argument (null, misaligned, inconsistent sizes) */
  PA_ERR_UNSUPPORTED = -2, /* valid but not built: head_dim, dtype or group size  */
  PA_ERR_CUDA = -3,        /* a CUDA runtime call or kernel launch failed          */
  PA_ERR_DEVICE = -4,      /* pa_device_status found a flagged device-side problem */
  PA_ERR_NO_BLOCKS = -5    /* block manager: no free or evictable block left       */
};

/* bits of the device status word */
enum {
  PA_DEV_BAD_SLOT = 1,        /* append: slot >= num_blocks*16 (row skipped)          */
  PA_DEV_BAD_BLOCK_ID = 2,    /* a block-table entry outside [0, num_blocks) (skipped) */
  PA_DEV_BAD_CONTEXT = 4,     /* context_len < 0 or > max_blocks_per_seq*16 (clamped) */
  PA_DEV_WAIT_TIMEOUT = 8,    /* a bounded wait on a copy barrier gave up              */
  PA_DEV_BAD_POSITION = 16,   /* RoPE: position outside [0, max_positions) (row skipped) */
  PA_DEV_RANGE = 32           /* INT8 prompt pass: a value past fp16's range (clamped) */
};

/* Geometry of the KV pool, shared by every call. */
typedef struct {
  int num_blocks;   /* physical blocks in each of k_pool and v_pool (>= 1)   */
  int num_kv_heads; /* H_kv (>= 1)                                            */
  int block_size;   /* tokens per block; must be PA_BLOCK_SIZE (16)          */
  int head_dim;     /* D: 64 or 128                                           */
  int dtype;        /* pa_dtype of pools, q, k_new/v_new and out; PA_I8 for  */
                    /* an INT8 cache (the *_int8 calls; q and out then have  */
                    /* their own act_dtype)                                  */
} pa_pool_desc;

/* Library version (PA_VERSION of the build). */
PA_API int pa_version(void);

/* Message for the last non-OK return on the calling thread ("" if none).
 * The pointer stays valid until the next pa_* call on that thread. */
PA_API const char* pa_last_error(void);

/*
 * pa_append_kv -- write this step's new K/V rows into the pool.
 *
 * The per-step in-place KV write ("Mini inference engine", step 2: append on
 * each step; "LLM Inference Server", Stage 1: new K/V slices written into
 * pre-allocated buffers in place), routed through a slot mapping into the
 * 16-token block pool.  For every token t with slot = slot_mapping[t] >= 0:
 *     k_pool[slot/16][h][slot%16][:] = k_new[t][h][:]   for all h,
 * and the same for V.  A negative slot skips the token (padding).  The copy is
 * bit-exact.  Slots must be distinct; with duplicates the surviving row is
 * unspecified.
 *
 *   k_pool, v_pool : [num_blocks][H_kv][16][D], written in place
 *   slot_mapping   : int64 [num_tokens]
 *   k_new, v_new   : [num_tokens][H_kv][D]
 *   num_tokens     : >= 0 (0 is a no-op)
 * Errors: PA_ERR_INVALID for null pointers, pointers not 16-byte aligned,
 * block_size != 16, num_tokens < 0; PA_ERR_UNSUPPORTED for other head_dim or
 * dtype.  A slot >= num_blocks*16 is skipped and sets PA_DEV_BAD_SLOT.
 */
PA_API int pa_append_kv(void* k_pool, void* v_pool, const int64_t* slot_mapping,
                 const void* k_new, const void* v_new, int num_tokens,
                 const pa_pool_desc* pool, void* stream);

/*
 * pa_decode_workspace_size -- bytes of device scratch pa_decode_attention
 * needs for the split-K partials of this batch shape (0 when no sequence can
 * span more than one partition).  partition_size as in pa_decode_attention.
 * Returns 0 and sets pa_last_error on invalid arguments.
 */
PA_API size_t pa_decode_workspace_size(int num_seqs, int num_q_heads, int max_context_len,
                                int partition_size, const pa_pool_desc* pool);

/* The partition (tokens per split-K unit) that pa_decode_attention will use
 * for this shape: partition_size itself when nonzero, else the automatic
 * choice.  The automatic choice takes the smallest partition of at least 256
 * tokens whose (sequence, KV head, partition) units all fit one resident wave
 * of the current device (3 decode CTAs per SM, the SM count queried from the
 * device); when even 2048-token partitions overflow a wave it takes 1024.
 * With no device current (planning on a host without a GPU) it assumes a full
 * GB300's 152 SMs.  pa_decode_workspace_size follows the same choice, so
 * size the workspace with the device that will run the call current. */
PA_API int pa_decode_partition_size(int num_seqs, int max_context_len, int partition_size,
                             const pa_pool_desc* pool);

/* The automatic choice above for a device of sm_count SMs (e.g. to plan for a
 * partition of a GPU).  Returns 0 and sets pa_last_error on invalid arguments
 * (sm_count < 1, a bad pool). */
PA_API int pa_decode_partition_size_on(int num_seqs, int max_context_len, int partition_size,
                                       const pa_pool_desc* pool, int sm_count);

/*
 * pa_decode_attention -- one query token per sequence over its paged cache.
 *
 * For each sequence s and q head h (KV head g = h / G):
 *     out[s][h] = softmax_i( scale * q[s][h] . K_s[i][g] ) V_s[i][g],  i < context_lens[s]
 * where K_s / V_s are the sequence's blocks read through its block table
 * (decode passes only the newly sampled token, "LLM Inference Server", Stage 1;
 * the fused attention kernel with GQA of "LLM Inference Server From Scratch",
 * How it works, 4).  A sequence with context_len 0 gets a zero row.
 *
 * Work is split into partitions of `partition_size` tokens (split-K); a
 * sequence spanning several partitions has its partial softmax results merged
 * by log-sum-exp, by whichever of its partitions finishes last (one kernel).
 * The result does not depend on the partition beyond fp32 rounding.
 *
 *   out               : [num_seqs][num_q_heads][D], written
 *   q                 : [num_seqs][num_q_heads][D]
 *   k_pool, v_pool    : pool layout above, read only
 *   block_tables      : int32 [num_seqs][max_blocks_per_seq]
 *   context_lens      : int32 [num_seqs], each in [0, max_context_len]
 *   scale             : softmax scale (e.g. 1/sqrt(D)), finite
 *   max_context_len   : host-known upper bound of context_lens (sizes the grid;
 *                       no device-to-host copy is made)
 *   partition_size    : tokens per split-K unit: 0 = automatic, else a multiple
 *                       of 16 in [16, 2048]
 *   workspace         : device scratch of >= pa_decode_workspace_size(...) bytes,
 *                       16-byte aligned (may be NULL when that size is 0).  Its
 *                       first 256 KiB hold split-K completion counters that must
 *                       be zero when a call starts: zero-fill the buffer once
 *                       before its first use; every call that completes leaves
 *                       them zero again, whatever shapes the calls have.  After
 *                       a PA_DEV_WAIT_TIMEOUT report, zero-fill it again.  Two
 *                       calls in flight at once must not share a workspace.
 * Errors: PA_ERR_INVALID for null or misaligned pointers, num_q_heads not a
 * multiple of num_kv_heads, max_context_len > max_blocks_per_seq*16, a bad
 * partition_size, a too-small workspace or a non-finite scale;
 * PA_ERR_UNSUPPORTED for head_dim not 64/128, G > 8, a pool too large for
 * 32-bit row coordinates, or split-K over more than 65536 (sequence, KV head)
 * pairs in one call.
 */
PA_API int pa_decode_attention(void* out, const void* q, const void* k_pool, const void* v_pool,
                        const int32_t* block_tables, const int32_t* context_lens,
                        float scale, int num_seqs, int num_q_heads, int max_blocks_per_seq,
                        int max_context_len, int partition_size, const pa_pool_desc* pool,
                        void* workspace, size_t workspace_bytes, void* stream);

/*
 * pa_decode_step -- one decode step in one launch: pa_append_kv of every
 * sequence's new token followed by pa_decode_attention.
 *
 * In a decode step each sequence gains exactly one token, at position
 * context_lens[s] - 1 (its slot comes from the block table, so no slot
 * mapping is passed); k_new / v_new hold those tokens, [num_seqs][H_kv][D] in
 * the pool dtype, 16-byte aligned.  The CTA that attends to a sequence's last
 * partition writes the token (K and V, its KV head) into the pool before it
 * reads that block, so the result equals pa_append_kv at those slots followed
 * by pa_decode_attention, bit for bit, and the pool keeps the token for the
 * next step.  A sequence with context_len 0 appends nothing.  Arguments,
 * workspace and errors as pa_decode_attention, plus PA_ERR_INVALID for null or
 * misaligned k_new / v_new.
 */
PA_API int pa_decode_step(void* out, const void* q, void* k_pool, void* v_pool, const void* k_new,
                          const void* v_new, const int32_t* block_tables, const int32_t* context_lens,
                          float scale, int num_seqs, int num_q_heads, int max_blocks_per_seq,
                          int max_context_len, int partition_size, const pa_pool_desc* pool,
                          void* workspace, size_t workspace_bytes, void* stream);

/*
 * pa_verify_attention -- attention for the verification pass of speculative
 * decoding: q_len query tokens per sequence (the last accepted token and the
 * q_len - 1 drafted ones, "LLM Inference Server", Batched Scheduling &
 * Speculative Decoding: the target model checks K = 4 drafted tokens in one
 * forward pass, so q_len = K + 1 = 5), all already appended to the pool.
 * Query i of sequence s sits at position p = context_lens[s] - q_len + i and
 * attends keys 0..p (causal), exactly as a prompt pass over a cached prefix
 * would; q_len = 1 is pa_decode_attention.  The K/V blocks are read once for
 * all q_len x G query rows of a KV head, and long contexts are split into
 * pieces merged by log-sum-exp as in pa_decode_attention.  At head dim 128 the
 * pieces are the stream-K ranges of a persistent launch (one CTA per SM, each
 * range at least partition_size tokens of work, 1024 when partition_size is
 * 0); at head dim 64 they are partitions of partition_size tokens.
 *
 *   out, q        : [num_seqs][q_len][num_q_heads][D], bf16 or fp16 pools
 *   context_lens  : int32 [num_seqs], each >= q_len (rows whose position is
 *                   negative see no key and are zero)
 *   workspace     : >= pa_verify_workspace_size(...) bytes, with the zero-fill
 *                   contract of pa_decode_attention
 * Errors as pa_decode_attention, plus PA_ERR_INVALID for q_len < 1 and
 * PA_ERR_UNSUPPORTED for fp32 pools or (num_q_heads/num_kv_heads) * q_len > 32.
 */
PA_API size_t pa_verify_workspace_size(int num_seqs, int q_len, int num_q_heads, int max_context_len,
                                       int partition_size, const pa_pool_desc* pool);
PA_API int pa_verify_attention(void* out, const void* q, const void* k_pool, const void* v_pool,
                               const int32_t* block_tables, const int32_t* context_lens, float scale,
                               int num_seqs, int q_len, int num_q_heads, int max_blocks_per_seq,
                               int max_context_len, int partition_size, const pa_pool_desc* pool,
                               void* workspace, size_t workspace_bytes, void* stream);

/*
 * pa_prefill_attention -- the causal prompt pass over the same pool.
 *
 * Prefill processes all prompt tokens at once (q_len = prompt length,
 * "LLM Inference Server", Stage 1) under a causal mask ("LLM Inference Server
 * From Scratch", What you build / How it works, 4).  Sequence s owns query
 * rows cu_q_lens[s] .. cu_q_lens[s+1]-1; its K/V (prompt tokens already
 * appended) are the first context_lens[s] positions of its blocks.  Query i of
 * the sequence sits at position p = context_lens[s] - q_len_s + i and attends
 * keys 0..p, so a cached prefix (context_len > q_len) is handled too.
 *
 *   out, q        : [cu_q_lens[num_seqs]][num_q_heads][D]
 *   block_tables  : int32 [num_seqs][max_blocks_per_seq]
 *   cu_q_lens     : int32 [num_seqs+1], non-decreasing, cu_q_lens[0] = 0
 *   context_lens  : int32 [num_seqs], context_lens[s] >= q_len_s
 *   max_q_len     : host-known max of q_len_s (sizes the grid)
 *   max_context_len : host-known max of context_lens (<= max_blocks_per_seq*16)
 * Errors as pa_decode_attention; fp32 pools are PA_ERR_UNSUPPORTED here (the
 * prompt pass runs on bf16/fp16 tensor cores), as is a call with more than
 * ~2^31 (query tile, sequence, head) items.
 * Scheduling: the (query tile, head pair) items are handed out at run time
 * from a pair of device counters owned by the library.  Each call takes the
 * next of 1024 pairs per device in turn, and the call's last CTA sets its pair
 * back to zero.  Calls may overlap on different streams as long as fewer than
 * 1024 prompt passes (of this and the INT8 entry point) are in flight at once
 * on one device.  A call captured into a CUDA graph keeps the pair it drew at
 * capture: replays of one graph run one after another, not concurrently.
 */
PA_API int pa_prefill_attention(void* out, const void* q, const void* k_pool, const void* v_pool,
                         const int32_t* block_tables, const int32_t* cu_q_lens,
                         const int32_t* context_lens, float scale, int num_seqs,
                         int num_q_heads, int max_blocks_per_seq, int max_q_len,
                         int max_context_len, const pa_pool_desc* pool, void* stream);

/*
 * INT8 KV cache ("LLM Inference Server", Optional Bonus Extensions: INT8
 * KV-Cache Quantization -- the cached K and V are quantised dynamically to
 * int8 per token head; the quantiser is the symmetric absmax rule of its
 * Required Mathematical Concepts: s = max|x| / 127, x_q = round(x / s),
 * x_hat = s * x_q).
 *
 * Storage, with pool->dtype = PA_I8:
 *   k_codes, v_codes   : int8    [num_blocks][H_kv][16][D]  (the float pool layout)
 *   k_scales, v_scales : float32 [num_blocks][H_kv][16]     (one per row)
 * Row (block, head, offset) stands for x_hat[d] = scales[row] * codes[row][d].
 * q, out, k_new and v_new have the activation dtype `act_dtype`, PA_BF16 or
 * PA_F16.  Pointers: codes and k_new/v_new/q/out 16-byte aligned, scales
 * 16-byte aligned, slot_mapping 8-byte aligned.
 */

/*
 * pa_append_kv_int8 -- quantise this step's new K/V rows into the INT8 cache.
 *
 * For every token t with slot = slot_mapping[t] >= 0 and every KV head h, the
 * row x = k_new[t][h][:] (act_dtype values, widened exactly to float32) is
 * stored as
 *     s = max_d |x[d]| / 127                     (float32, IEEE division)
 *     k_codes[slot/16][h][slot%16][d] = round(x[d] / s)   (IEEE division,
 *                                                  ties to even, in [-127, 127])
 *     k_scales[slot/16][h][slot%16]   = s
 * and the same for V; an all-zero row stores s = 0 and zero codes.  Codes and
 * scales are bit-exact functions of the row (every float operation is a single
 * correctly rounded one).  A row holding Inf or NaN stores unspecified codes
 * and a non-finite scale.  Negative slots are skipped; slots must be distinct.
 * Errors as pa_append_kv, plus PA_ERR_INVALID when pool->dtype is not PA_I8 or
 * act_dtype is not PA_BF16/PA_F16.
 */
PA_API int pa_append_kv_int8(void* k_codes, void* v_codes, float* k_scales, float* v_scales,
                             const int64_t* slot_mapping, const void* k_new, const void* v_new,
                             int num_tokens, int act_dtype, const pa_pool_desc* pool, void* stream);

/*
 * pa_decode_attention_int8 -- pa_decode_attention over an INT8 cache.
 *
 * out[s][h] = softmax_i( scale * q[s][h] . K_hat_s[i][g] ) V_hat_s[i][g] with
 * K_hat = k_scales * k_codes and V_hat = v_scales * v_codes row by row; every
 * other rule (GQA mapping, context lengths, zero rows, split-K partitions and
 * their merge, the workspace and its zero-fill contract, partition_size) is
 * that of pa_decode_attention, with pool->dtype = PA_I8 in
 * pa_decode_workspace_size / pa_decode_partition_size.  Scores, softmax and
 * accumulation run in fp32; out (act_dtype) is rounded once.  Scale entries
 * of positions outside the contexts are never used, whatever they hold.
 * Errors as pa_decode_attention, plus PA_ERR_INVALID when pool->dtype is not
 * PA_I8 or act_dtype is not PA_BF16/PA_F16.
 */
PA_API int pa_decode_attention_int8(void* out, const void* q, const void* k_codes,
                                    const void* v_codes, const float* k_scales,
                                    const float* v_scales, const int32_t* block_tables,
                                    const int32_t* context_lens, float scale, int num_seqs,
                                    int num_q_heads, int max_blocks_per_seq, int max_context_len,
                                    int partition_size, int act_dtype, const pa_pool_desc* pool,
                                    void* workspace, size_t workspace_bytes, void* stream);

/*
 * pa_verify_attention_int8 -- pa_verify_attention over an INT8 cache: q_len
 * query tokens per sequence (the last accepted token and the drafted ones of
 * "LLM Inference Server", Batched Scheduling & Speculative Decoding), query i
 * at position context_lens[s] - q_len + i attending the dequantised keys
 * 0..that position, as pa_decode_attention_int8 does for one query.  The code
 * and scale blocks of a KV head are read once for all q_len x G query rows;
 * long contexts split into partitions of partition_size tokens merged by
 * log-sum-exp.  q_len = 1 is pa_decode_attention_int8.
 *
 *   out, q        : [num_seqs][q_len][num_q_heads][D], act_dtype
 *   context_lens  : rows whose position is negative see no key and are zero
 *   workspace     : >= pa_verify_workspace_size(..., pool) bytes with
 *                   pool->dtype = PA_I8, zero-filled before its first use
 * Errors as pa_decode_attention_int8, plus PA_ERR_INVALID for q_len < 1 and
 * PA_ERR_UNSUPPORTED for (num_q_heads/num_kv_heads) * q_len > 32.
 */
PA_API int pa_verify_attention_int8(void* out, const void* q, const void* k_codes,
                                    const void* v_codes, const float* k_scales,
                                    const float* v_scales, const int32_t* block_tables,
                                    const int32_t* context_lens, float scale, int num_seqs,
                                    int q_len, int num_q_heads, int max_blocks_per_seq,
                                    int max_context_len, int partition_size, int act_dtype,
                                    const pa_pool_desc* pool, void* workspace,
                                    size_t workspace_bytes, void* stream);

/*
 * pa_prefill_attention_int8 -- pa_prefill_attention over an INT8 cache: the
 * causal prompt pass (all prompt tokens at once, "LLM Inference Server",
 * Stage 1) with keys and values x_hat = scales[row] * codes[row][d].  The
 * pass is compute-bound, so each sequence's blocks of its first
 * context_lens[s] positions are first dequantised into `workspace` (every
 * x_hat rounded once to fp16, 11 significant bits, in the float pool layout),
 * and the fp16 prompt pass runs over those copies; bf16 queries are converted
 * to fp16 in shared memory by the pass (exactly, within fp16's range) and the
 * output rows stored as bf16.
 *   out, q   : act_dtype [cu_q_lens[num_seqs]][num_q_heads][D]
 *   the other arguments as pa_prefill_attention; pool->dtype = PA_I8
 *   workspace: device, 16-byte aligned, >= pa_prefill_int8_workspace_size()
 *              bytes, owned by the caller, its contents scratch: the fp16 K
 *              and V copies of num_seqs x ceil(max_context_len / 16) blocks
 *              (each 256-byte aligned) and their int32 block table.
 * Errors as pa_prefill_attention, plus PA_ERR_INVALID for a missing or small
 * workspace and PA_ERR_UNSUPPORTED past 65535 sequences.  A block id outside
 * the pool sets PA_DEV_BAD_BLOCK_ID and its keys read as zeros; a cache or
 * query value past fp16's range (|x| > 65504 for a dequantised cache value,
 * |q| >= 65536 for a bf16 query, inf and NaN included) is clamped to +-65504
 * and sets PA_DEV_RANGE.
 * pa_prefill_int8_workspace_size returns 0 (and sets the last error) for a
 * pool that is not INT8 or negative sizes.
 */
PA_API size_t pa_prefill_int8_workspace_size(int num_seqs, int max_context_len,
                                             const pa_pool_desc* pool);
PA_API int pa_prefill_attention_int8(void* out, const void* q, const void* k_codes,
                                     const void* v_codes, const float* k_scales,
                                     const float* v_scales, const int32_t* block_tables,
                                     const int32_t* cu_q_lens, const int32_t* context_lens,
                                     float scale, int num_seqs, int num_q_heads,
                                     int max_blocks_per_seq, int max_q_len, int max_context_len,
                                     int act_dtype, const pa_pool_desc* pool, void* workspace,
                                     size_t workspace_bytes, void* stream);

/*
 * Rotary position embedding fused into the append.  The pages name RoPE as a
 * step to fuse with attention ("Mini inference engine", Story / portfolio:
 * fuse qkv_proj + RoPE + attention) without defining it; this is the
 * half-split rotary embedding of the Llama family: for position p, entries j
 * and j + D/2 of a row (j < D/2) turn by the angle p * theta^(-2j/D):
 *     x'[j] = x[j] cos - x[j + D/2] sin,   x'[j + D/2] = x[j + D/2] cos + x[j] sin.
 *
 * pa_rope_cache -- fill cos_sin, float32 [max_positions][head_dim/2][2] =
 * (cos, sin) of p * theta^(-2j/head_dim), angles and trigonometry in float64,
 * stored rounded to float32.  Build it once per model; the calls below read
 * it.  Errors: PA_ERR_INVALID for a null or misaligned (8-byte) table,
 * max_positions < 0 or theta <= 0; PA_ERR_UNSUPPORTED for head_dim not 64/128.
 */
PA_API int pa_rope_cache(float* cos_sin, int max_positions, int head_dim, double theta, void* stream);

/*
 * pa_append_kv_rope -- pa_append_kv with every K row rotated at its token's
 * position (positions: int32 [num_tokens]) on the way into the pool: fp32
 * arithmetic on the table entries, one rounding to the pool dtype.  V rows are
 * copied bit for bit.  A position outside [0, max_positions) skips the token's
 * K rows and sets PA_DEV_BAD_POSITION.  Errors as pa_append_kv, plus
 * PA_ERR_INVALID for a null positions or cos_sin pointer.
 */
PA_API int pa_append_kv_rope(void* k_pool, void* v_pool, const int64_t* slot_mapping, const int32_t* positions,
                             const void* k_new, const void* v_new, int num_tokens, const float* cos_sin,
                             int max_positions, const pa_pool_desc* pool, void* stream);

/*
 * pa_apply_rope -- rotate rows x [num_tokens][num_heads][head_dim] (dtype
 * PA_F32/PA_BF16/PA_F16) in place at their token's position: the queries of a
 * step, before pa_decode_attention / pa_verify_attention.
 */
PA_API int pa_apply_rope(void* x, const int32_t* positions, int num_tokens, int num_heads, int head_dim,
                         int dtype, const float* cos_sin, int max_positions, void* stream);

/*
 * Block manager with a prefix cache (host side).  The paged pool of 16-token
 * blocks reached through per-sequence block tables ("LLM Inference Server",
 * Optional Bonus Extensions: Paged KV-Cache Block Allocator; "LLM Inference
 * Server From Scratch", How it works, 3 Block Manager), with the hash-keyed
 * prefix cache of "LLM Inference Server", Stage 1 (a shared system prompt's KV
 * stored once and reused; hit/miss tracking).  The manager only does the
 * bookkeeping: it hands out slots (for pa_append_kv and friends), block tables
 * (for the attention calls) and copy-on-write pairs (for pa_copy_blocks).
 *
 * Policies, deterministic: full blocks are keyed by FNV-1a 64 over the
 * little-endian bytes of (parent block key, 16 token ids), content checked on
 * a hit; a prompt reuses its cached full blocks from the start up to the first
 * miss; new full blocks are cached at once; appending into a last block that
 * another table holds copies it first; freeing releases blocks last to first,
 * cached ones onto a least-recently-released list; allocation takes the
 * lowest free id, else evicts the least recently released cached block.  A
 * call that runs out of blocks returns PA_ERR_NO_BLOCKS and changes nothing.
 * A manager is not thread-safe.
 */
typedef struct pa_block_manager pa_block_manager;

typedef struct {
  int64_t hit_blocks;     /* prompt blocks found in the prefix cache            */
  int64_t miss_blocks;    /* full prompt blocks not found                       */
  int64_t cow_copies;     /* copy-on-write pairs handed out                      */
  int64_t evictions;      /* cached idle blocks reused for new data              */
  int32_t free_blocks;    /* never used or released uncached                    */
  int32_t cached_free_blocks; /* released, still cached, evictable             */
  int32_t used_blocks;    /* held by at least one table                         */
} pa_bm_stats;

/* A manager for num_blocks blocks, tables of up to max_blocks_per_seq
 * entries, sequence ids 0..max_seqs-1.  NULL on bad arguments. */
PA_API pa_block_manager* pa_bm_create(int num_blocks, int max_blocks_per_seq, int max_seqs);
PA_API void pa_bm_destroy(pa_block_manager* bm);

/* Start sequence `seq` with prompt token ids [prompt_len].  slots (int64
 * [prompt_len], host) receives the pool slot of every prompt position; the
 * return value (>= 0) is the number of leading prompt tokens whose blocks came
 * from the prefix cache (their K/V are already in the pool), else an error. */
PA_API int pa_bm_add_sequence(pa_block_manager* bm, int seq, const int32_t* prompt, int prompt_len,
                              int64_t* slots);

/* Append n tokens to `seq`: slots (int64 [n], host) receives their pool
 * slots.  When the sequence's last block is shared with another table it is
 * copied first: the pair (source block, new block) goes to copies (int32,
 * room for max_copies pairs; at most one pair per call) and *num_copies is
 * set; the caller runs pa_copy_blocks before writing the new tokens. */
PA_API int pa_bm_append(pa_block_manager* bm, int seq, const int32_t* tokens, int n, int64_t* slots,
                        int32_t* copies, int max_copies, int* num_copies);

/* One decode step: token tokens[i] appended to sequence seq_ids[i] for i < n
 * (distinct sequences), in order, all or nothing.  slots: int64 [n];
 * copy-on-write pairs (at most one per sequence) go to copies, in call
 * order.  The same result as n single-token pa_bm_append calls. */
PA_API int pa_bm_append_step(pa_block_manager* bm, const int32_t* seq_ids, const int32_t* tokens, int n,
                             int64_t* slots, int32_t* copies, int max_copies, int* num_copies);

/* `child` shares every block of `parent` (e.g. several samples of one prompt). */
PA_API int pa_bm_fork(pa_block_manager* bm, int parent, int child);

/* End `seq` and release its blocks. */
PA_API int pa_bm_free_sequence(pa_block_manager* bm, int seq);

/* Block tables (int32 [n][max_blocks], unused entries 0) and context lengths
 * (int32 [n]) of the listed live sequences, in host memory. */
PA_API int pa_bm_block_tables(const pa_block_manager* bm, const int32_t* seq_ids, int n, int32_t* tables,
                              int max_blocks, int32_t* context_lens);

PA_API int pa_bm_get_stats(const pa_block_manager* bm, pa_bm_stats* out);

/*
 * pa_copy_blocks -- copy whole pool blocks (every KV head, K and V) for
 * copy-on-write: pairs (int32 [num_pairs][2], DEVICE) = (source, destination)
 * block ids, destinations distinct and not sources.  Bit-exact.  Ids outside
 * the pool are skipped and set PA_DEV_BAD_BLOCK_ID.  Float pools only.
 */
PA_API int pa_copy_blocks(void* k_pool, void* v_pool, const int32_t* pairs, int num_pairs,
                          const pa_pool_desc* pool, void* stream);

/*
 * pa_copy_blocks_int8 -- pa_copy_blocks for an INT8 cache (pool->dtype =
 * PA_I8): copies the code blocks of K and V and, with them, the blocks' rows
 * of the K and V scale arrays (H_kv x 16 floats per block), so that the
 * destination block dequantises to exactly the source's values (the prefix
 * cache of "LLM Inference Server", Stage 1, over the INT8 cache of its
 * Optional Bonus Extensions).  Bit-exact.  Pointers 16-byte aligned, pairs
 * 8-byte aligned; ids outside the pool are skipped and set
 * PA_DEV_BAD_BLOCK_ID.  Errors: PA_ERR_INVALID when pool->dtype is not PA_I8.
 */
PA_API int pa_copy_blocks_int8(void* k_codes, void* v_codes, float* k_scales, float* v_scales,
                               const int32_t* pairs, int num_pairs, const pa_pool_desc* pool, void* stream);

/* Bytes of the per-device array behind pa_decode_attention_noalloc. */
#define PA_NOALLOC_SCRATCH_BYTES (32u << 20)

/*
 * pa_decode_attention_noalloc -- pa_decode_attention for callers that cannot
 * allocate device memory.  (The method as described has no counterpart: this
 * entry point exists for callers, not for the method.)
 *
 * Some callers cannot call cudaMalloc: a serving loop that may not allocate
 * once it is running, an embedder that hands over only tensors it already
 * owns, a plain C host without a device allocator.  This call takes the same
 * arguments as pa_decode_attention minus the workspace and allocates nothing;
 * the split-K partials go to a file-scope device array of
 * PA_NOALLOC_SCRATCH_BYTES (32 MiB) that every GPU loading the library holds
 * until the process exits.  The caller still passes every input and output.
 *  - A shape whose partials need more than PA_NOALLOC_SCRATCH_BYTES
 *    (see pa_decode_workspace_size) returns PA_ERR_INVALID with a message,
 *    before anything is enqueued.  A larger partition_size needs less.
 *  - The first call on a device that needs the array looks up its device
 *    address (cudaGetSymbolAddress) with that device current; make that first
 *    call before any stream capture.  The address is remembered with the
 *    CUDA context it belongs to: after a device reset the next call looks it
 *    up again (so that call, too, should come before any capture).
 *  - Every call on a device shares the array and it keeps the last call's
 *    contents.  The split-K completion counters at its start must be zero
 *    when a call begins: each call clears the ones it uses (an asynchronous
 *    memset on `stream`) before its kernel.  Calls that overlap on the GPU
 *    (e.g. on two streams) race on it: serialise them.
 * Other errors as pa_decode_attention.
 */
PA_API int pa_decode_attention_noalloc(void* out, const void* q, const void* k_pool,
                                       const void* v_pool, const int32_t* block_tables,
                                       const int32_t* context_lens, float scale, int num_seqs,
                                       int num_q_heads, int max_blocks_per_seq,
                                       int max_context_len, int partition_size,
                                       const pa_pool_desc* pool, void* stream);

/*
 * pa_device_status -- read and clear the device status word of the current
 * device (bits PA_DEV_*).  Synchronises `stream` first.  Returns PA_OK when the
 * word was 0, PA_ERR_DEVICE when any bit was set (the bits are stored in
 * *status), PA_ERR_CUDA if the read failed.
 */
PA_API int pa_device_status(int* status, void* stream);

#ifdef __cplusplus
}
#endif

#endif /* PA_H_ */
