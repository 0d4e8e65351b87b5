// pa_api.cu -- the C ABI of libpa (declared in include/pa.h).
//
// Host side only: argument checks (all before anything is enqueued, so a bad
// call never reaches the GPU -- the idea of rejecting invalid requests before
// touching the GPU, "LLM Inference Server", Stage 4 input validation), the
// split-K partition choice, TMA descriptors for the KV pool, and the kernel
// launches.  No allocation, no synchronisation.
#include <cudaTypedefs.h>

#include <cmath>
#include <cstdarg>
#include <cstdio>
#include <cstring>
#include <mutex>
#include <string>

#include "pa.h"
#include "pa_internal.h"

// Device status word (PA_DEV_* bits), one per device that loads the library.
__device__ int g_pa_status = 0;
// Work counters of the prompt pass's run-time schedule: kSchedSlots pairs
// (items taken, CTAs finished), zero at load; each launch draws the next
// pair in turn and its last CTA sets the pair back to zero.
constexpr int kSchedSlots = 1024;
__device__ int g_pa_prefill_sched[2 * kSchedSlots] = {};

namespace {

// SMs assumed by the sizing calls when no device is current (a full GB300,
// the part sm_103a code runs on); with a device current its own count is used.
constexpr int kDefaultSms = 152;
// Decode CTAs resident on one SM at once (three 64 KB stage sets), and the
// smallest partition the automatic choice uses: below it the split-K merge
// costs more than it hides.
constexpr int kCtasPerSm = 3;
constexpr int kMinPartition = 256;
constexpr int kMaxPartition = 2048;   // 32 blocks per warp of a 4-warp CTA
// Split-K completion counters occupy a fixed region at the start of the
// workspace, so no shape's partials ever overlap another shape's counters.
constexpr int kMaxCounters = 65536;   // (sequence, KV head) pairs per split-K call
constexpr size_t kCounterBytes = kMaxCounters * sizeof(int);

thread_local std::string t_err;

int fail(int code, const char* fmt, ...) {
  char buf[512];
  va_list ap;
  va_start(ap, fmt);
  vsnprintf(buf, sizeof(buf), fmt, ap);
  va_end(ap);
  t_err = buf;
  return code;
}

int cuda_fail(cudaError_t e, const char* what) {
  return fail(PA_ERR_CUDA, "%s: %s", what, cudaGetErrorString(e));
}

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

int elem_bytes(int dtype) {
  switch (dtype) {
    case PA_F32: return 4;
    case PA_BF16:
    case PA_F16: return 2;
    case PA_I8: return 1;
    default: return 0;
  }
}

// The float entry points take float pools only; an INT8 cache has its own.
int reject_int8(const pa_pool_desc* pool) {
  if (pool->dtype == PA_I8)
    return fail(PA_ERR_INVALID, "an INT8 pool (dtype PA_I8) needs the *_int8 entry points");
  return PA_OK;
}

int check_int8(const pa_pool_desc* pool, int act_dtype) {
  if (pool->dtype != PA_I8) return fail(PA_ERR_INVALID, "pool dtype must be PA_I8 for an INT8 cache");
  if (act_dtype != PA_BF16 && act_dtype != PA_F16)
    return fail(PA_ERR_INVALID, "act_dtype must be PA_BF16 or PA_F16 (got %d)", act_dtype);
  return PA_OK;
}

int check_pool(const pa_pool_desc* pool) {
  if (!pool) return fail(PA_ERR_INVALID, "pool descriptor is NULL");
  if (pool->block_size != PA_BLOCK_SIZE)
    return fail(PA_ERR_INVALID, "block_size must be %d (got %d)", PA_BLOCK_SIZE, pool->block_size);
  if (pool->num_blocks < 1) return fail(PA_ERR_INVALID, "num_blocks must be >= 1");
  if (pool->num_kv_heads < 1) return fail(PA_ERR_INVALID, "num_kv_heads must be >= 1");
  if (elem_bytes(pool->dtype) == 0) return fail(PA_ERR_UNSUPPORTED, "dtype %d not supported", pool->dtype);
  if (pool->head_dim != 64 && pool->head_dim != 128)
    return fail(PA_ERR_UNSUPPORTED, "head_dim %d not supported (64 or 128)", pool->head_dim);
  if (static_cast<long long>(pool->num_blocks) * pool->num_kv_heads * PA_BLOCK_SIZE > 0x7fffffffLL)
    return fail(PA_ERR_UNSUPPORTED, "pool too large for 32-bit row coordinates");
  return PA_OK;
}

int* status_ptr() {
  static std::mutex mu;
  static int* cache[64] = {};
  static void* cache_ctx[64] = {};
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return nullptr;
  std::lock_guard<std::mutex> lock(mu);
  if (!cache[dev] || cache_ctx[dev] != pa::current_context()) {
    void* p = nullptr;
    if (cudaGetSymbolAddress(&p, g_pa_status) != cudaSuccess) return nullptr;
    cache[dev] = static_cast<int*>(p);
    // the lookup made the device's primary context current if none was
    cache_ctx[dev] = pa::current_context();
  }
  return cache[dev];
}

// This launch's pair of schedule counters on the current device, or null.
// Launches take the pairs in turn, so two launches share a pair only when
// kSchedSlots launches of the prompt pass are in flight at once.
int* prefill_sched_ptr() {
  static std::mutex mu;
  static int* cache[64] = {};
  static void* cache_ctx[64] = {};
  static unsigned next_slot[64] = {};
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return nullptr;
  std::lock_guard<std::mutex> lock(mu);
  if (!cache[dev] || cache_ctx[dev] != pa::current_context()) {
    void* p = nullptr;
    if (cudaGetSymbolAddress(&p, g_pa_prefill_sched) != cudaSuccess) return nullptr;
    cache[dev] = static_cast<int*>(p);
    cache_ctx[dev] = pa::current_context();
  }
  const unsigned slot = next_slot[dev]++ % kSchedSlots;
  return cache[dev] + 2 * slot;
}

// SMs of the current device, or kDefaultSms when none is current.
int current_sms() {
  const int n = pa::device_sm_count();
  return n > 0 ? n : kDefaultSms;
}

// ctas_per_sm: CTAs of the kernel resident on one SM; past_wave: the
// partition when not even 2048-token partitions fit one wave.
int choose_partition_on(int num_seqs, int num_kv_heads, int max_context_len, int requested, int sms,
                        int ctas_per_sm = kCtasPerSm, int past_wave = 1024) {
  if (requested > 0) return requested;
  // One resident wave when the batch allows it: the largest partition count
  // (smallest partition, not below kMinPartition) whose (sequence, KV head,
  // partition) units all fit on the GPU at once.  Past that the decode runs in
  // several waves of past_wave-token partitions.
  const long long wave = static_cast<long long>(ctas_per_sm) * (sms > 0 ? sms : kDefaultSms);
  const auto units = [&](int p) {
    return static_cast<long long>(num_seqs) * num_kv_heads * ((max_context_len + p - 1) / p);
  };
  if (units(kMaxPartition) > wave) return past_wave;
  int p = kMaxPartition;
  while (p > kMinPartition && units(p / 2) <= wave) p /= 2;
  return p;
}

int choose_partition(int num_seqs, int num_kv_heads, int max_context_len, int requested) {
  return choose_partition_on(num_seqs, num_kv_heads, max_context_len, requested,
                             requested > 0 ? kDefaultSms : current_sms());
}

// The INT8 kernel with more than one 8-column query tile (a verification pass
// of G * q_len > 8 query columns) holds more accumulators: 2 CTAs per SM, and
// each CTA pays a fixed start-up (its query tiles widened and scaled, their
// bias products, a merge of every column), so when the batch does not fit one
// wave it takes the longest partitions (measured on the Llama-3-8B-shaped
// batch-64 pass of 4 drafts: 471 / 307 / 225 / 194 us at 256 / 512 / 1024 /
// 2048 tokens).
bool int8_wide(int num_q_heads, int q_len, const pa_pool_desc* pool) {
  return pool->dtype == PA_I8 && q_len > 1 && (num_q_heads / pool->num_kv_heads) * q_len > 8;
}

int choose_partition_for(int num_seqs, int num_q_heads, int q_len, int max_context_len, int requested,
                         const pa_pool_desc* pool) {
  if (!int8_wide(num_q_heads, q_len, pool)) return choose_partition(num_seqs, pool->num_kv_heads, max_context_len, requested);
  return choose_partition_on(num_seqs, pool->num_kv_heads, max_context_len, requested,
                             requested > 0 ? kDefaultSms : current_sms(), 2, kMaxPartition);
}

int max_splits_for(int max_context_len, int part_blocks) {
  const int nblk = (max_context_len + PA_BLOCK_SIZE - 1) / PA_BLOCK_SIZE;
  return nblk == 0 ? 1 : (nblk + part_blocks - 1) / part_blocks;
}

size_t align256(size_t x) { return (x + 255) & ~static_cast<size_t>(255); }

// Verification on the tensor-core kernel: a float pool, head dim 128 and more
// than one query position.
bool verify_on_umma(int q_len, const pa_pool_desc* pool) {
  return q_len > 1 && pool->head_dim == 128 && pool->dtype != PA_I8;
}

// Partial-output slots per query row of a verify call: the split-K partitions of
// the mma.sync kernels, or the stream-K segments of the tensor-core kernel.
int verify_slots(int q_len, const pa_pool_desc* pool, int max_context_len, int part_blocks) {
  return verify_on_umma(q_len, pool) ? pa::verify_umma_slots(max_context_len, part_blocks)
                                     : max_splits_for(max_context_len, part_blocks);
}

// [counters: kCounterBytes][partial outputs: rows x D fp32][partial lse: rows fp32]
struct WsLayout {
  size_t o_off, lse_off, total;
};

WsLayout ws_layout(int num_seqs, int num_q_heads, int max_splits, int head_dim) {
  WsLayout w{0, 0, 0};
  if (max_splits <= 1) return w;
  const size_t rows = static_cast<size_t>(num_seqs) * num_q_heads * max_splits;
  w.o_off = kCounterBytes;
  w.lse_off = align256(w.o_off + rows * head_dim * sizeof(float));
  w.total = w.lse_off + rows * sizeof(float);
  return w;
}

// ---- TMA descriptors of the pool ---------------------------------------------

PFN_cuTensorMapEncodeTiled_v12000 encode_fn() {
  static PFN_cuTensorMapEncodeTiled_v12000 fn = [] {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) !=
            cudaSuccess ||
        q != cudaDriverEntryPointSuccess)
      return static_cast<PFN_cuTensorMapEncodeTiled_v12000>(nullptr);
    return reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(p);
  }();
  return fn;
}

// The pool viewed as a 2-D tensor of rows (block, head, offset) x head_dim.
// bf16/fp16: boxes of 16 rows x 64 elements (128 bytes), 128-byte swizzle.
// INT8 codes: boxes of 16 whole rows (D bytes), 128-byte swizzle for D = 128
// and 64-byte swizzle for D = 64.
int make_pool_map(CUtensorMap* map, const void* pool_ptr, const pa_pool_desc* pool) {
  auto enc = encode_fn();
  if (!enc) return fail(PA_ERR_CUDA, "cuTensorMapEncodeTiled is not available from the driver");
  const bool q8 = pool->dtype == PA_I8;
  const CUtensorMapDataType dt = q8 ? CU_TENSOR_MAP_DATA_TYPE_UINT8
                                    : (pool->dtype == PA_BF16 ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16
                                                              : CU_TENSOR_MAP_DATA_TYPE_FLOAT16);
  cuuint64_t dims[2] = {static_cast<cuuint64_t>(pool->head_dim),
                        static_cast<cuuint64_t>(pool->num_blocks) * pool->num_kv_heads * PA_BLOCK_SIZE};
  cuuint64_t strides[1] = {static_cast<cuuint64_t>(pool->head_dim) * elem_bytes(pool->dtype)};
  cuuint32_t box[2] = {q8 ? static_cast<cuuint32_t>(pool->head_dim) : 64u, PA_BLOCK_SIZE};
  cuuint32_t estr[2] = {1, 1};
  const CUtensorMapSwizzle sw =
      (q8 && pool->head_dim == 64) ? CU_TENSOR_MAP_SWIZZLE_64B : CU_TENSOR_MAP_SWIZZLE_128B;
  CUresult r = enc(map, dt, 2, const_cast<void*>(pool_ptr), dims, strides, box, estr,
                   CU_TENSOR_MAP_INTERLEAVE_NONE, sw, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                   CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  if (r != CUDA_SUCCESS) return fail(PA_ERR_CUDA, "cuTensorMapEncodeTiled failed (%d)", static_cast<int>(r));
  return PA_OK;
}

// The prompt-pass queries q [rows][H][D] viewed as a 3-D tensor (D, H, rows)
// for 128-row boxes of one head and 64 columns (128 bytes, 128-byte swizzle):
// one box is half of a query tile in the layout the S product reads.  `rows`
// is an upper bound of the query rows; the kernel loads by this map only
// whole 128-row tiles of a prompt, which lie inside the caller's buffer.
int make_q_map(CUtensorMap* map, const void* q, int dtype, int num_heads, int head_dim, long long rows) {
  auto enc = encode_fn();
  if (!enc) return fail(PA_ERR_CUDA, "cuTensorMapEncodeTiled is not available from the driver");
  const CUtensorMapDataType dt = dtype == PA_BF16 ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16 : CU_TENSOR_MAP_DATA_TYPE_FLOAT16;
  cuuint64_t dims[3] = {static_cast<cuuint64_t>(head_dim), static_cast<cuuint64_t>(num_heads),
                        static_cast<cuuint64_t>(rows)};
  cuuint64_t strides[2] = {static_cast<cuuint64_t>(head_dim) * 2,
                           static_cast<cuuint64_t>(num_heads) * head_dim * 2};
  cuuint32_t box[3] = {64u, 1u, 128u};
  cuuint32_t estr[3] = {1, 1, 1};
  CUresult r = enc(map, dt, 3, const_cast<void*>(q), dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
                   CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  if (r != CUDA_SUCCESS) return fail(PA_ERR_CUDA, "cuTensorMapEncodeTiled (queries) failed (%d)", static_cast<int>(r));
  return PA_OK;
}

// Small per-thread cache: encoding is cheap but not free, and the same pools
// are passed on every step.
struct MapEntry {
  const void* ptr;
  pa_pool_desc desc;
  CUtensorMap map;
  bool used;
};

int pool_map(CUtensorMap* out, const void* ptr, const pa_pool_desc* pool) {
  thread_local MapEntry cache[8] = {};
  thread_local int next = 0;
  for (auto& e : cache) {
    if (e.used && e.ptr == ptr && std::memcmp(&e.desc, pool, sizeof(pa_pool_desc)) == 0) {
      *out = e.map;
      return PA_OK;
    }
  }
  MapEntry& e = cache[next];
  next = (next + 1) % 8;
  const int rc = make_pool_map(&e.map, ptr, pool);
  if (rc != PA_OK) {
    e.used = false;
    return rc;
  }
  e.ptr = ptr;
  e.desc = *pool;
  e.used = true;
  *out = e.map;
  return PA_OK;
}

int check_decode_shape(int num_seqs, int num_q_heads, int max_blocks_per_seq, int max_context_len,
                       int partition_size, const pa_pool_desc* pool) {
  int rc = check_pool(pool);
  if (rc != PA_OK) return rc;
  if (num_seqs < 0) return fail(PA_ERR_INVALID, "num_seqs must be >= 0");
  if (num_seqs > 65535) return fail(PA_ERR_UNSUPPORTED, "num_seqs > 65535");
  if (num_q_heads < 1 || num_q_heads % pool->num_kv_heads != 0)
    return fail(PA_ERR_INVALID, "num_q_heads (%d) must be a positive multiple of num_kv_heads (%d)",
                num_q_heads, pool->num_kv_heads);
  if (num_q_heads / pool->num_kv_heads > 8)
    return fail(PA_ERR_UNSUPPORTED, "query group size %d > 8", num_q_heads / pool->num_kv_heads);
  if (pool->num_kv_heads > 65535) return fail(PA_ERR_UNSUPPORTED, "num_kv_heads > 65535");
  if (max_context_len < 0) return fail(PA_ERR_INVALID, "max_context_len must be >= 0");
  if (max_blocks_per_seq < 0) return fail(PA_ERR_INVALID, "max_blocks_per_seq must be >= 0");
  if (static_cast<long long>(max_context_len) > static_cast<long long>(max_blocks_per_seq) * PA_BLOCK_SIZE)
    return fail(PA_ERR_INVALID, "max_context_len %d exceeds max_blocks_per_seq*16 = %lld", max_context_len,
                static_cast<long long>(max_blocks_per_seq) * PA_BLOCK_SIZE);
  if (partition_size != 0 &&
      (partition_size < PA_BLOCK_SIZE || partition_size > kMaxPartition || partition_size % PA_BLOCK_SIZE))
    return fail(PA_ERR_INVALID, "partition_size %d must be 0 or a multiple of 16 in [16, %d]", partition_size,
                kMaxPartition);
  return PA_OK;
}

}  // namespace

namespace pa {
int set_last_error(int code, const char* msg) {
  t_err = msg;
  return code;
}

void* current_context() {
  using GetCurrent = CUresult (*)(CUcontext*);
  static GetCurrent fn = [] {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuCtxGetCurrent", &p, 12000, cudaEnableDefault, &q) != cudaSuccess ||
        q != cudaDriverEntryPointSuccess)
      return static_cast<GetCurrent>(nullptr);
    return reinterpret_cast<GetCurrent>(p);
  }();
  CUcontext c = nullptr;
  if (!fn || fn(&c) != CUDA_SUCCESS) return nullptr;
  return c;
}

int device_sm_count() {
  static std::mutex mu;
  static int cache[64] = {};
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return 0;
  std::lock_guard<std::mutex> lock(mu);
  if (cache[dev] == 0) {
    int n = 0;
    if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) return 0;
    cache[dev] = n;
  }
  return cache[dev];
}
}  // namespace pa

extern "C" {

int pa_version(void) { return PA_VERSION; }

const char* pa_last_error(void) { return t_err.c_str(); }

int pa_append_kv(void* k_pool, void* v_pool, const int64_t* slot_mapping, const void* k_new,
                 const void* v_new, int num_tokens, const pa_pool_desc* pool, void* stream) {
  t_err.clear();
  int rc = check_pool(pool);
  if (rc != PA_OK) return rc;
  if ((rc = reject_int8(pool)) != PA_OK) return rc;
  if (num_tokens < 0) return fail(PA_ERR_INVALID, "num_tokens must be >= 0");
  if (num_tokens == 0) return PA_OK;
  if (!k_pool || !v_pool || !slot_mapping || !k_new || !v_new)
    return fail(PA_ERR_INVALID, "null pointer argument");
  if (!aligned16(k_pool) || !aligned16(v_pool) || !aligned16(k_new) || !aligned16(v_new))
    return fail(PA_ERR_INVALID, "pools and k_new/v_new must be 16-byte aligned");
  if ((reinterpret_cast<uintptr_t>(slot_mapping) & 7u) != 0)
    return fail(PA_ERR_INVALID, "slot_mapping must be 8-byte aligned");
  const int row_bytes = pool->head_dim * elem_bytes(pool->dtype);
  int* status = status_ptr();
  if (!status) return fail(PA_ERR_CUDA, "no CUDA device / status word unavailable");
  cudaError_t e = pa::launch_append(k_pool, v_pool, slot_mapping, k_new, v_new, num_tokens,
                                    pool->num_kv_heads, row_bytes, pool->num_blocks, status,
                                    static_cast<cudaStream_t>(stream));
  if (e != cudaSuccess) return cuda_fail(e, "append_kv launch");
  return PA_OK;
}

int pa_decode_partition_size(int num_seqs, int max_context_len, int partition_size,
                             const pa_pool_desc* pool) {
  t_err.clear();
  if (check_pool(pool) != PA_OK) return 0;
  return choose_partition(num_seqs, pool->num_kv_heads, max_context_len, partition_size);
}

int pa_decode_partition_size_on(int num_seqs, int max_context_len, int partition_size,
                                const pa_pool_desc* pool, int sm_count) {
  t_err.clear();
  if (check_pool(pool) != PA_OK) return 0;
  if (sm_count < 1) {
    fail(PA_ERR_INVALID, "sm_count must be >= 1");
    return 0;
  }
  return choose_partition_on(num_seqs, pool->num_kv_heads, max_context_len, partition_size, sm_count);
}

size_t pa_decode_workspace_size(int num_seqs, int num_q_heads, int max_context_len, int partition_size,
                                const pa_pool_desc* pool) {
  t_err.clear();
  const int mb = (max_context_len + PA_BLOCK_SIZE - 1) / PA_BLOCK_SIZE;
  if (check_decode_shape(num_seqs, num_q_heads, mb, max_context_len, partition_size, pool) != PA_OK) return 0;
  const int p = choose_partition(num_seqs, pool->num_kv_heads, max_context_len, partition_size);
  const int ms = max_splits_for(max_context_len, p / PA_BLOCK_SIZE);
  return ws_layout(num_seqs, num_q_heads, ms, pool->head_dim).total;
}

namespace {
int decode_impl(void* out, const void* q, const void* k_pool, const void* v_pool, const void* k_new,
                const void* v_new, const int32_t* block_tables, const int32_t* context_lens, float scale,
                int num_seqs, int num_q_heads, int max_blocks_per_seq, int max_context_len, int partition_size,
                const pa_pool_desc* pool, void* workspace, size_t workspace_bytes, void* stream);
}

int pa_decode_attention(void* out, const void* q, const void* k_pool, const void* v_pool,
                        const int32_t* block_tables, const int32_t* context_lens, float scale,
                        int num_seqs, int num_q_heads, int max_blocks_per_seq, int max_context_len,
                        int partition_size, const pa_pool_desc* pool, void* workspace,
                        size_t workspace_bytes, void* stream) {
  t_err.clear();
  return decode_impl(out, q, k_pool, v_pool, nullptr, nullptr, block_tables, context_lens, scale, num_seqs,
                     num_q_heads, max_blocks_per_seq, max_context_len, partition_size, pool, workspace,
                     workspace_bytes, stream);
}

int pa_decode_step(void* out, const void* q, void* k_pool, void* v_pool, const void* k_new, const void* v_new,
                   const int32_t* block_tables, const int32_t* context_lens, float scale, int num_seqs,
                   int num_q_heads, int max_blocks_per_seq, int max_context_len, int partition_size,
                   const pa_pool_desc* pool, void* workspace, size_t workspace_bytes, void* stream) {
  t_err.clear();
  if (num_seqs > 0 && (!k_new || !v_new)) return fail(PA_ERR_INVALID, "null k_new / v_new");
  if (num_seqs > 0 && (!aligned16(k_new) || !aligned16(v_new)))
    return fail(PA_ERR_INVALID, "k_new / v_new must be 16-byte aligned");
  return decode_impl(out, q, k_pool, v_pool, k_new, v_new, block_tables, context_lens, scale, num_seqs,
                     num_q_heads, max_blocks_per_seq, max_context_len, partition_size, pool, workspace,
                     workspace_bytes, stream);
}

namespace {
int decode_impl(void* out, const void* q, const void* k_pool, const void* v_pool, const void* k_new,
                const void* v_new, const int32_t* block_tables, const int32_t* context_lens, float scale,
                int num_seqs, int num_q_heads, int max_blocks_per_seq, int max_context_len, int partition_size,
                const pa_pool_desc* pool, void* workspace, size_t workspace_bytes, void* stream) {
  int rc = check_decode_shape(num_seqs, num_q_heads, max_blocks_per_seq, max_context_len, partition_size, pool);
  if (rc != PA_OK) return rc;
  if ((rc = reject_int8(pool)) != PA_OK) return rc;
  if (!std::isfinite(scale)) return fail(PA_ERR_INVALID, "scale must be finite");
  if (num_seqs == 0) return PA_OK;
  if (!out || !q || !k_pool || !v_pool || !context_lens || (max_blocks_per_seq > 0 && !block_tables))
    return fail(PA_ERR_INVALID, "null pointer argument");
  if (!aligned16(out) || !aligned16(q) || !aligned16(k_pool) || !aligned16(v_pool))
    return fail(PA_ERR_INVALID, "out, q and the pools must be 16-byte aligned");
  if ((reinterpret_cast<uintptr_t>(block_tables) & 3u) || (reinterpret_cast<uintptr_t>(context_lens) & 3u))
    return fail(PA_ERR_INVALID, "block_tables and context_lens must be 4-byte aligned");

  const int part = choose_partition(num_seqs, pool->num_kv_heads, max_context_len, partition_size);
  const int part_blocks = part / PA_BLOCK_SIZE;
  const int max_splits = max_splits_for(max_context_len, part_blocks);
  const WsLayout ws = ws_layout(num_seqs, num_q_heads, max_splits, pool->head_dim);
  if (ws.total > 0 && static_cast<long long>(num_seqs) * pool->num_kv_heads > kMaxCounters)
    return fail(PA_ERR_UNSUPPORTED, "split-K over more than %d (sequence, KV head) pairs in one call",
                kMaxCounters);
  if (ws.total > 0) {
    if (!workspace) return fail(PA_ERR_INVALID, "workspace of %zu bytes required, got NULL", ws.total);
    if (workspace_bytes < ws.total)
      return fail(PA_ERR_INVALID, "workspace too small: %zu < %zu bytes", workspace_bytes, ws.total);
    if (!aligned16(workspace)) return fail(PA_ERR_INVALID, "workspace must be 16-byte aligned");
  }
  int* status = status_ptr();
  if (!status) return fail(PA_ERR_CUDA, "no CUDA device / status word unavailable");

  pa::DecodeArgs a{};
  a.out = out;
  a.q = q;
  a.k_pool = k_pool;
  a.v_pool = v_pool;
  a.block_tables = block_tables;
  a.context_lens = context_lens;
  a.scale_log2 = scale * 1.4426950408889634f;
  a.num_seqs = num_seqs;
  a.num_q_heads = num_q_heads;
  a.num_kv_heads = pool->num_kv_heads;
  a.head_dim = pool->head_dim;
  a.max_blocks_per_seq = max_blocks_per_seq;
  a.max_context_len = max_context_len;
  a.num_blocks = pool->num_blocks;
  a.part_blocks = part_blocks;
  a.max_splits = max_splits;
  a.ws_count = ws.total ? static_cast<int*>(workspace) : nullptr;
  a.ws_o = ws.total ? reinterpret_cast<float*>(static_cast<char*>(workspace) + ws.o_off) : nullptr;
  a.ws_lse = ws.total ? reinterpret_cast<float*>(static_cast<char*>(workspace) + ws.lse_off) : nullptr;
  a.status = status;
  a.q_len = 1;
  a.k_new = k_new;
  a.v_new = v_new;
  cudaStream_t st = static_cast<cudaStream_t>(stream);

  cudaError_t e;
  if (pool->dtype == PA_F32) {
    e = pa::launch_decode_simt(a, pool->dtype, st);
  } else {
    CUtensorMap kmap, vmap;
    if ((rc = pool_map(&kmap, k_pool, pool)) != PA_OK) return rc;
    if ((rc = pool_map(&vmap, v_pool, pool)) != PA_OK) return rc;
    e = pa::launch_decode_tc(a, pool->dtype, kmap, vmap, st);
  }
  if (e != cudaSuccess) return cuda_fail(e, "decode launch");
  return PA_OK;
}
}  // namespace

size_t pa_verify_workspace_size(int num_seqs, int q_len, int num_q_heads, int max_context_len, int partition_size,
                                const pa_pool_desc* pool) {
  t_err.clear();
  const int mb = (max_context_len + PA_BLOCK_SIZE - 1) / PA_BLOCK_SIZE;
  if (check_decode_shape(num_seqs, num_q_heads, mb, max_context_len, partition_size, pool) != PA_OK) return 0;
  if (q_len < 1) {
    fail(PA_ERR_INVALID, "q_len must be >= 1");
    return 0;
  }
  const int p = choose_partition_for(num_seqs, num_q_heads, q_len, max_context_len, partition_size, pool);
  const int ms = verify_slots(q_len, pool, max_context_len, p / PA_BLOCK_SIZE);
  return ws_layout(num_seqs * q_len, num_q_heads, ms, pool->head_dim).total;
}

int pa_verify_attention(void* out, const void* q, const void* k_pool, const void* v_pool,
                        const int32_t* block_tables, const int32_t* context_lens, float scale, int num_seqs,
                        int q_len, int num_q_heads, int max_blocks_per_seq, int max_context_len,
                        int partition_size, const pa_pool_desc* pool, void* workspace, size_t workspace_bytes,
                        void* stream) {
  t_err.clear();
  int rc = check_decode_shape(num_seqs, num_q_heads, max_blocks_per_seq, max_context_len, partition_size, pool);
  if (rc != PA_OK) return rc;
  if ((rc = reject_int8(pool)) != PA_OK) return rc;
  if (pool->dtype == PA_F32) return fail(PA_ERR_UNSUPPORTED, "verify needs bf16 or fp16 pools");
  if (q_len < 1) return fail(PA_ERR_INVALID, "q_len must be >= 1");
  if ((num_q_heads / pool->num_kv_heads) * q_len > 32)
    return fail(PA_ERR_UNSUPPORTED, "query group x q_len = %d > 32", (num_q_heads / pool->num_kv_heads) * q_len);
  if (static_cast<long long>(num_seqs) * q_len > 0x7fffffffLL) return fail(PA_ERR_UNSUPPORTED, "too many rows");
  if (!std::isfinite(scale)) return fail(PA_ERR_INVALID, "scale must be finite");
  if (num_seqs == 0) return PA_OK;
  if (!out || !q || !k_pool || !v_pool || !context_lens || (max_blocks_per_seq > 0 && !block_tables))
    return fail(PA_ERR_INVALID, "null pointer argument");
  if (!aligned16(out) || !aligned16(q) || !aligned16(k_pool) || !aligned16(v_pool))
    return fail(PA_ERR_INVALID, "out, q and the pools must be 16-byte aligned");
  if ((reinterpret_cast<uintptr_t>(block_tables) & 3u) || (reinterpret_cast<uintptr_t>(context_lens) & 3u))
    return fail(PA_ERR_INVALID, "block_tables and context_lens must be 4-byte aligned");

  const int part = choose_partition(num_seqs, pool->num_kv_heads, max_context_len, partition_size);
  const int part_blocks = part / PA_BLOCK_SIZE;
  const int max_splits = verify_slots(q_len, pool, max_context_len, part_blocks);
  const WsLayout ws = ws_layout(num_seqs * q_len, num_q_heads, max_splits, pool->head_dim);
  if (ws.total > 0 && static_cast<long long>(num_seqs) * pool->num_kv_heads > kMaxCounters)
    return fail(PA_ERR_UNSUPPORTED, "split-K over more than %d (sequence, KV head) pairs in one call",
                kMaxCounters);
  if (ws.total > 0) {
    if (!workspace) return fail(PA_ERR_INVALID, "workspace of %zu bytes required, got NULL", ws.total);
    if (workspace_bytes < ws.total)
      return fail(PA_ERR_INVALID, "workspace too small: %zu < %zu bytes", workspace_bytes, ws.total);
    if (!aligned16(workspace)) return fail(PA_ERR_INVALID, "workspace must be 16-byte aligned");
  }
  int* status = status_ptr();
  if (!status) return fail(PA_ERR_CUDA, "no CUDA device / status word unavailable");

  pa::DecodeArgs a{};
  a.out = out;
  a.q = q;
  a.k_pool = k_pool;
  a.v_pool = v_pool;
  a.block_tables = block_tables;
  a.context_lens = context_lens;
  a.scale_log2 = scale * 1.4426950408889634f;
  a.num_seqs = num_seqs;
  a.num_q_heads = num_q_heads;
  a.num_kv_heads = pool->num_kv_heads;
  a.head_dim = pool->head_dim;
  a.max_blocks_per_seq = max_blocks_per_seq;
  a.max_context_len = max_context_len;
  a.num_blocks = pool->num_blocks;
  a.part_blocks = part_blocks;
  a.max_splits = max_splits;
  a.ws_count = ws.total ? static_cast<int*>(workspace) : nullptr;
  a.ws_o = ws.total ? reinterpret_cast<float*>(static_cast<char*>(workspace) + ws.o_off) : nullptr;
  a.ws_lse = ws.total ? reinterpret_cast<float*>(static_cast<char*>(workspace) + ws.lse_off) : nullptr;
  a.status = status;
  a.q_len = q_len;
  CUtensorMap kmap, vmap;
  if ((rc = pool_map(&kmap, k_pool, pool)) != PA_OK) return rc;
  if ((rc = pool_map(&vmap, v_pool, pool)) != PA_OK) return rc;
  const cudaStream_t st = static_cast<cudaStream_t>(stream);
  cudaError_t e = q_len == 1                                 ? pa::launch_decode_tc(a, pool->dtype, kmap, vmap, st)
                  : verify_on_umma(q_len, pool) ? pa::launch_verify_umma(a, pool->dtype, kmap, vmap, st)
                                                            : pa::launch_verify_tc(a, pool->dtype, kmap, vmap, st);
  if (e != cudaSuccess) return cuda_fail(e, "verify launch");
  return PA_OK;
}

namespace {

// The prompt pass over a bf16/fp16 pool once the call has been validated: q
// and the output rows in act_dtype (the pool's type, or bf16 over an fp16
// pool).
int prefill_launch(void* out, const void* q, const void* k_pool, const void* v_pool, const int32_t* block_tables,
                   const int32_t* cu_q_lens, const int32_t* context_lens, float scale, int num_seqs,
                   int num_q_heads, int max_blocks_per_seq, int max_q_len, const pa_pool_desc* pool, int act_dtype,
                   int* status, void* stream) {
  pa::PrefillArgs a{};
  a.out = out;
  a.q = q;
  a.block_tables = block_tables;
  a.cu_q_lens = cu_q_lens;
  a.context_lens = context_lens;
  a.scale_log2 = scale * 1.4426950408889634f;
  a.num_seqs = num_seqs;
  a.num_q_heads = num_q_heads;
  a.num_kv_heads = pool->num_kv_heads;
  a.head_dim = pool->head_dim;
  a.max_blocks_per_seq = max_blocks_per_seq;
  a.num_blocks = pool->num_blocks;
  a.max_q_len = max_q_len;
  a.status = status;
  a.sched = prefill_sched_ptr();
  if (!a.sched) return fail(PA_ERR_CUDA, "no CUDA device / schedule counters unavailable");
  CUtensorMap kmap, vmap, qmap;
  int rc;
  if ((rc = pool_map(&kmap, k_pool, pool)) != PA_OK) return rc;
  if ((rc = pool_map(&vmap, v_pool, pool)) != PA_OK) return rc;
  if ((rc = make_q_map(&qmap, q, act_dtype, num_q_heads, pool->head_dim,
                       static_cast<long long>(num_seqs) * max_q_len)) != PA_OK)
    return rc;
  cudaError_t e =
      pa::launch_prefill_umma(a, pool->dtype, act_dtype, kmap, vmap, qmap, static_cast<cudaStream_t>(stream));
  if (e != cudaSuccess) return cuda_fail(e, "prefill launch");
  return PA_OK;
}

// Checks shared by the prompt passes (pool already checked): returns PA_OK, or
// the error of the first violated rule.  Sets *nothing when there is no work.
int check_prefill_args(const void* out, const void* q, const int32_t* block_tables, const int32_t* cu_q_lens,
                       const int32_t* context_lens, float scale, int num_seqs, int num_q_heads, int max_q_len,
                       int max_context_len, bool* nothing) {
  *nothing = false;
  if (!std::isfinite(scale)) return fail(PA_ERR_INVALID, "scale must be finite");
  if (max_q_len < 0 || max_q_len > max_context_len)
    return fail(PA_ERR_INVALID, "max_q_len %d must be in [0, max_context_len=%d]", max_q_len, max_context_len);
  if (num_seqs == 0 || max_q_len == 0) {
    *nothing = true;
    return PA_OK;
  }
  if (!out || !q || !block_tables || !cu_q_lens || !context_lens) return fail(PA_ERR_INVALID, "null pointer argument");
  if (!aligned16(out) || !aligned16(q)) return fail(PA_ERR_INVALID, "out and q must be 16-byte aligned");
  if ((reinterpret_cast<uintptr_t>(block_tables) & 3u) || (reinterpret_cast<uintptr_t>(cu_q_lens) & 3u) ||
      (reinterpret_cast<uintptr_t>(context_lens) & 3u))
    return fail(PA_ERR_INVALID, "int32 arrays must be 4-byte aligned");
  if ((max_q_len + 63) / 64 > 0x7fffffff) return fail(PA_ERR_UNSUPPORTED, "max_q_len too large");
  // the run-time schedule counts (query tile, sequence, head) items in int32
  if (static_cast<long long>((max_q_len + 127) / 128) * num_seqs * num_q_heads > 0x7fff0000LL)
    return fail(PA_ERR_UNSUPPORTED, "too many query tiles in one prompt pass");
  return PA_OK;
}

// Workspace of the INT8 prompt pass: the fp16 copies of the K and V blocks
// (num_seqs * B blocks, B = blocks of max_context_len) and their block table.
struct PrefillQ8Ws {
  size_t k_off, v_off, table_off, total;
  int B;
};

PrefillQ8Ws prefill_q8_ws(int num_seqs, int max_context_len, const pa_pool_desc* pool) {
  PrefillQ8Ws w{0, 0, 0, 0, 0};
  w.B = (max_context_len + PA_BLOCK_SIZE - 1) / PA_BLOCK_SIZE;
  const size_t blocks = static_cast<size_t>(num_seqs) * w.B;
  if (blocks == 0) return w;
  const size_t pool_bytes = blocks * pool->num_kv_heads * PA_BLOCK_SIZE * pool->head_dim * 2;
  w.k_off = 0;
  w.v_off = align256(pool_bytes);
  w.table_off = w.v_off + align256(pool_bytes);
  w.total = w.table_off + blocks * sizeof(int32_t);
  return w;
}

}  // namespace

int pa_prefill_attention(void* out, const void* q, const void* k_pool, const void* v_pool,
                         const int32_t* block_tables, const int32_t* cu_q_lens, const int32_t* context_lens,
                         float scale, int num_seqs, int num_q_heads, int max_blocks_per_seq, int max_q_len,
                         int max_context_len, const pa_pool_desc* pool, void* stream) {
  t_err.clear();
  int rc = check_decode_shape(num_seqs, num_q_heads, max_blocks_per_seq, max_context_len, 0, pool);
  if (rc != PA_OK) return rc;
  if ((rc = reject_int8(pool)) != PA_OK) return rc;
  if (pool->dtype == PA_F32) return fail(PA_ERR_UNSUPPORTED, "prefill needs bf16 or fp16 pools");
  bool nothing;
  if ((rc = check_prefill_args(out, q, block_tables, cu_q_lens, context_lens, scale, num_seqs, num_q_heads, max_q_len,
                               max_context_len, &nothing)) != PA_OK)
    return rc;
  if (nothing) return PA_OK;
  if (!k_pool || !v_pool) return fail(PA_ERR_INVALID, "null pointer argument");
  if (!aligned16(k_pool) || !aligned16(v_pool)) return fail(PA_ERR_INVALID, "the pools must be 16-byte aligned");
  int* status = status_ptr();
  if (!status) return fail(PA_ERR_CUDA, "no CUDA device / status word unavailable");
  return prefill_launch(out, q, k_pool, v_pool, block_tables, cu_q_lens, context_lens, scale, num_seqs, num_q_heads,
                        max_blocks_per_seq, max_q_len, pool, pool->dtype, status, stream);
}

size_t pa_prefill_int8_workspace_size(int num_seqs, int max_context_len, const pa_pool_desc* pool) {
  t_err.clear();
  if (check_pool(pool) != PA_OK) return 0;
  if (pool->dtype != PA_I8) {
    fail(PA_ERR_INVALID, "the INT8 prompt pass needs an INT8 pool");
    return 0;
  }
  if (num_seqs < 0 || max_context_len < 0) {
    fail(PA_ERR_INVALID, "num_seqs and max_context_len must be >= 0");
    return 0;
  }
  return prefill_q8_ws(num_seqs, max_context_len, pool).total;
}

int pa_prefill_attention_int8(void* out, const void* q, const void* k_codes, const void* v_codes,
                              const float* k_scales, const float* v_scales, const int32_t* block_tables,
                              const int32_t* cu_q_lens, const int32_t* context_lens, float scale, int num_seqs,
                              int num_q_heads, int max_blocks_per_seq, int max_q_len, int max_context_len,
                              int act_dtype, const pa_pool_desc* pool, void* workspace, size_t workspace_bytes,
                              void* stream) {
  t_err.clear();
  int rc = check_decode_shape(num_seqs, num_q_heads, max_blocks_per_seq, max_context_len, 0, pool);
  if (rc != PA_OK) return rc;
  if ((rc = check_int8(pool, act_dtype)) != PA_OK) return rc;
  bool nothing;
  if ((rc = check_prefill_args(out, q, block_tables, cu_q_lens, context_lens, scale, num_seqs, num_q_heads, max_q_len,
                               max_context_len, &nothing)) != PA_OK)
    return rc;
  if (nothing) return PA_OK;
  if (num_seqs > 65535) return fail(PA_ERR_UNSUPPORTED, "more than 65535 sequences in one INT8 prompt pass");
  if (static_cast<long long>(num_seqs) * ((max_context_len + PA_BLOCK_SIZE - 1) / PA_BLOCK_SIZE) > 0x7fffffffLL)
    return fail(PA_ERR_UNSUPPORTED, "num_seqs x context blocks too large");
  if (!k_codes || !v_codes || !k_scales || !v_scales) return fail(PA_ERR_INVALID, "null pointer argument");
  if (!aligned16(k_codes) || !aligned16(v_codes) || !aligned16(k_scales) || !aligned16(v_scales))
    return fail(PA_ERR_INVALID, "codes and scales must be 16-byte aligned");
  const PrefillQ8Ws ws = prefill_q8_ws(num_seqs, max_context_len, pool);
  if (!workspace) return fail(PA_ERR_INVALID, "workspace of %zu bytes required, got NULL", ws.total);
  if (workspace_bytes < ws.total)
    return fail(PA_ERR_INVALID, "workspace too small: %zu < %zu bytes", workspace_bytes, ws.total);
  if (!aligned16(workspace)) return fail(PA_ERR_INVALID, "workspace must be 16-byte aligned");
  int* status = status_ptr();
  if (!status) return fail(PA_ERR_CUDA, "no CUDA device / status word unavailable");
  const cudaStream_t st = static_cast<cudaStream_t>(stream);
  char* base = static_cast<char*>(workspace);
  int32_t* table = reinterpret_cast<int32_t*>(base + ws.table_off);
  // the pass runs in fp16 over the copies; bf16 queries are converted in
  // shared memory and the output rows stored as bf16 by the pass itself
  pa::DequantQ8Args dq{};
  dq.k_codes = static_cast<const int8_t*>(k_codes);
  dq.v_codes = static_cast<const int8_t*>(v_codes);
  dq.k_scales = k_scales;
  dq.v_scales = v_scales;
  dq.block_tables = block_tables;
  dq.context_lens = context_lens;
  dq.num_seqs = num_seqs;
  dq.max_blocks_per_seq = max_blocks_per_seq;
  dq.num_kv_heads = pool->num_kv_heads;
  dq.head_dim = pool->head_dim;
  dq.num_blocks = pool->num_blocks;
  dq.B = ws.B;
  dq.k_out = base + ws.k_off;
  dq.v_out = base + ws.v_off;
  dq.table_out = table;
  dq.status = status;
  cudaError_t e = pa::launch_dequant_q8(dq, st);
  if (e != cudaSuccess) return cuda_fail(e, "INT8 prompt-pass dequantisation launch");
  const pa_pool_desc fpool{num_seqs * ws.B, pool->num_kv_heads, pool->block_size, pool->head_dim, PA_F16};
  return prefill_launch(out, q, base + ws.k_off, base + ws.v_off, table, cu_q_lens, context_lens, scale, num_seqs,
                        num_q_heads, ws.B, max_q_len, &fpool, act_dtype, status, stream);
}

int pa_append_kv_int8(void* k_codes, void* v_codes, float* k_scales, float* v_scales,
                      const int64_t* slot_mapping, const void* k_new, const void* v_new, int num_tokens,
                      int act_dtype, const pa_pool_desc* pool, void* stream) {
  t_err.clear();
  int rc = check_pool(pool);
  if (rc != PA_OK) return rc;
  if ((rc = check_int8(pool, act_dtype)) != PA_OK) return rc;
  if (num_tokens < 0) return fail(PA_ERR_INVALID, "num_tokens must be >= 0");
  if (num_tokens == 0) return PA_OK;
  if (!k_codes || !v_codes || !k_scales || !v_scales || !slot_mapping || !k_new || !v_new)
    return fail(PA_ERR_INVALID, "null pointer argument");
  if (!aligned16(k_codes) || !aligned16(v_codes) || !aligned16(k_scales) || !aligned16(v_scales) ||
      !aligned16(k_new) || !aligned16(v_new))
    return fail(PA_ERR_INVALID, "codes, scales and k_new/v_new must be 16-byte aligned");
  if ((reinterpret_cast<uintptr_t>(slot_mapping) & 7u) != 0)
    return fail(PA_ERR_INVALID, "slot_mapping must be 8-byte aligned");
  int* status = status_ptr();
  if (!status) return fail(PA_ERR_CUDA, "no CUDA device / status word unavailable");
  cudaError_t e = pa::launch_append_q8(k_codes, v_codes, k_scales, v_scales, slot_mapping, k_new, v_new,
                                       num_tokens, pool->num_kv_heads, pool->head_dim, act_dtype,
                                       pool->num_blocks, status, static_cast<cudaStream_t>(stream));
  if (e != cudaSuccess) return cuda_fail(e, "append_kv_int8 launch");
  return PA_OK;
}

namespace {
// Decode (q_len = 1) and verification (q_len > 1) over an INT8 cache: one kernel
// family, split-K partitions of partition_size tokens.
int int8_attention(void* out, const void* q, const void* k_codes, const void* v_codes, const float* k_scales,
                   const float* v_scales, const int32_t* block_tables, const int32_t* context_lens, float scale,
                   int num_seqs, int q_len, int num_q_heads, int max_blocks_per_seq, int max_context_len,
                   int partition_size, int act_dtype, const pa_pool_desc* pool, void* workspace,
                   size_t workspace_bytes, void* stream) {
  int rc = check_decode_shape(num_seqs, num_q_heads, max_blocks_per_seq, max_context_len, partition_size, pool);
  if (rc != PA_OK) return rc;
  if ((rc = check_int8(pool, act_dtype)) != PA_OK) return rc;
  if (q_len < 1) return fail(PA_ERR_INVALID, "q_len must be >= 1");
  if ((num_q_heads / pool->num_kv_heads) * q_len > 32)
    return fail(PA_ERR_UNSUPPORTED, "query group x q_len = %d > 32", (num_q_heads / pool->num_kv_heads) * q_len);
  if (static_cast<long long>(num_seqs) * q_len > 0x7fffffffLL) return fail(PA_ERR_UNSUPPORTED, "too many rows");
  if (!std::isfinite(scale)) return fail(PA_ERR_INVALID, "scale must be finite");
  if (num_seqs == 0) return PA_OK;
  if (!out || !q || !k_codes || !v_codes || !k_scales || !v_scales || !context_lens ||
      (max_blocks_per_seq > 0 && !block_tables))
    return fail(PA_ERR_INVALID, "null pointer argument");
  if (!aligned16(out) || !aligned16(q) || !aligned16(k_codes) || !aligned16(v_codes) || !aligned16(k_scales) ||
      !aligned16(v_scales))
    return fail(PA_ERR_INVALID, "out, q, codes and scales must be 16-byte aligned");
  if ((reinterpret_cast<uintptr_t>(block_tables) & 3u) || (reinterpret_cast<uintptr_t>(context_lens) & 3u))
    return fail(PA_ERR_INVALID, "block_tables and context_lens must be 4-byte aligned");

  const int part = choose_partition_for(num_seqs, num_q_heads, q_len, max_context_len, partition_size, pool);
  const int part_blocks = part / PA_BLOCK_SIZE;
  const int max_splits = max_splits_for(max_context_len, part_blocks);
  const WsLayout ws = ws_layout(num_seqs * q_len, num_q_heads, max_splits, pool->head_dim);
  if (ws.total > 0 && static_cast<long long>(num_seqs) * pool->num_kv_heads > kMaxCounters)
    return fail(PA_ERR_UNSUPPORTED, "split-K over more than %d (sequence, KV head) pairs in one call",
                kMaxCounters);
  if (ws.total > 0) {
    if (!workspace) return fail(PA_ERR_INVALID, "workspace of %zu bytes required, got NULL", ws.total);
    if (workspace_bytes < ws.total)
      return fail(PA_ERR_INVALID, "workspace too small: %zu < %zu bytes", workspace_bytes, ws.total);
    if (!aligned16(workspace)) return fail(PA_ERR_INVALID, "workspace must be 16-byte aligned");
  }
  int* status = status_ptr();
  if (!status) return fail(PA_ERR_CUDA, "no CUDA device / status word unavailable");

  pa::DecodeArgs a{};
  a.out = out;
  a.q = q;
  a.k_pool = k_codes;
  a.v_pool = v_codes;
  a.k_scales = k_scales;
  a.v_scales = v_scales;
  a.block_tables = block_tables;
  a.context_lens = context_lens;
  a.scale_log2 = scale * 1.4426950408889634f;
  a.num_seqs = num_seqs;
  a.num_q_heads = num_q_heads;
  a.num_kv_heads = pool->num_kv_heads;
  a.head_dim = pool->head_dim;
  a.max_blocks_per_seq = max_blocks_per_seq;
  a.max_context_len = max_context_len;
  a.num_blocks = pool->num_blocks;
  a.part_blocks = part_blocks;
  a.max_splits = max_splits;
  a.ws_count = ws.total ? static_cast<int*>(workspace) : nullptr;
  a.ws_o = ws.total ? reinterpret_cast<float*>(static_cast<char*>(workspace) + ws.o_off) : nullptr;
  a.ws_lse = ws.total ? reinterpret_cast<float*>(static_cast<char*>(workspace) + ws.lse_off) : nullptr;
  a.status = status;
  a.q_len = q_len;
  CUtensorMap kmap, vmap;
  if ((rc = pool_map(&kmap, k_codes, pool)) != PA_OK) return rc;
  if ((rc = pool_map(&vmap, v_codes, pool)) != PA_OK) return rc;
  cudaError_t e = pa::launch_decode_q8(a, act_dtype, kmap, vmap, static_cast<cudaStream_t>(stream));
  if (e != cudaSuccess) return cuda_fail(e, q_len == 1 ? "decode_int8 launch" : "verify_int8 launch");
  return PA_OK;
}
}  // namespace

int pa_decode_attention_int8(void* out, const void* q, const void* k_codes, const void* v_codes,
                             const float* k_scales, const float* v_scales, const int32_t* block_tables,
                             const int32_t* context_lens, float scale, int num_seqs, int num_q_heads,
                             int max_blocks_per_seq, int max_context_len, int partition_size, int act_dtype,
                             const pa_pool_desc* pool, void* workspace, size_t workspace_bytes, void* stream) {
  t_err.clear();
  return int8_attention(out, q, k_codes, v_codes, k_scales, v_scales, block_tables, context_lens, scale, num_seqs,
                        1, num_q_heads, max_blocks_per_seq, max_context_len, partition_size, act_dtype, pool,
                        workspace, workspace_bytes, stream);
}

int pa_verify_attention_int8(void* out, const void* q, const void* k_codes, const void* v_codes,
                             const float* k_scales, const float* v_scales, const int32_t* block_tables,
                             const int32_t* context_lens, float scale, int num_seqs, int q_len, int num_q_heads,
                             int max_blocks_per_seq, int max_context_len, int partition_size, int act_dtype,
                             const pa_pool_desc* pool, void* workspace, size_t workspace_bytes, void* stream) {
  t_err.clear();
  return int8_attention(out, q, k_codes, v_codes, k_scales, v_scales, block_tables, context_lens, scale, num_seqs,
                        q_len, num_q_heads, max_blocks_per_seq, max_context_len, partition_size, act_dtype, pool,
                        workspace, workspace_bytes, stream);
}

int pa_rope_cache(float* cos_sin, int max_positions, int head_dim, double theta, void* stream) {
  t_err.clear();
  if (head_dim != 64 && head_dim != 128) return fail(PA_ERR_UNSUPPORTED, "head_dim %d not supported", head_dim);
  if (max_positions < 0) return fail(PA_ERR_INVALID, "max_positions must be >= 0");
  if (!(theta > 0.0) || !std::isfinite(theta)) return fail(PA_ERR_INVALID, "theta must be positive and finite");
  if (max_positions == 0) return PA_OK;
  if (!cos_sin || (reinterpret_cast<uintptr_t>(cos_sin) & 7u))
    return fail(PA_ERR_INVALID, "cos_sin must be a non-null 8-byte aligned pointer");
  cudaError_t e = pa::launch_rope_cache(cos_sin, max_positions, head_dim, theta, static_cast<cudaStream_t>(stream));
  if (e != cudaSuccess) return cuda_fail(e, "rope cache launch");
  return PA_OK;
}

int pa_append_kv_rope(void* k_pool, void* v_pool, const int64_t* slot_mapping, const int32_t* positions,
                      const void* k_new, const void* v_new, int num_tokens, const float* cos_sin, int max_positions,
                      const pa_pool_desc* pool, void* stream) {
  t_err.clear();
  int rc = check_pool(pool);
  if (rc != PA_OK) return rc;
  if ((rc = reject_int8(pool)) != PA_OK) return rc;
  if (num_tokens < 0) return fail(PA_ERR_INVALID, "num_tokens must be >= 0");
  if (max_positions < 0) return fail(PA_ERR_INVALID, "max_positions must be >= 0");
  if (num_tokens == 0) return PA_OK;
  if (!k_pool || !v_pool || !slot_mapping || !positions || !k_new || !v_new || !cos_sin)
    return fail(PA_ERR_INVALID, "null pointer argument");
  if (!aligned16(k_pool) || !aligned16(v_pool) || !aligned16(k_new) || !aligned16(v_new))
    return fail(PA_ERR_INVALID, "pools and k_new/v_new must be 16-byte aligned");
  if ((reinterpret_cast<uintptr_t>(slot_mapping) & 7u) || (reinterpret_cast<uintptr_t>(positions) & 3u) ||
      (reinterpret_cast<uintptr_t>(cos_sin) & 7u))
    return fail(PA_ERR_INVALID, "slot_mapping (8), positions (4) or cos_sin (8 bytes) misaligned");
  int* status = status_ptr();
  if (!status) return fail(PA_ERR_CUDA, "no CUDA device / status word unavailable");
  cudaError_t e = pa::launch_append_rope(k_pool, v_pool, slot_mapping, positions, k_new, v_new, cos_sin,
                                         max_positions, num_tokens, pool->num_kv_heads, pool->head_dim, pool->dtype,
                                         pool->num_blocks, status, static_cast<cudaStream_t>(stream));
  if (e != cudaSuccess) return cuda_fail(e, "append_kv_rope launch");
  return PA_OK;
}

int pa_apply_rope(void* x, const int32_t* positions, int num_tokens, int num_heads, int head_dim, int dtype,
                  const float* cos_sin, int max_positions, void* stream) {
  t_err.clear();
  if (head_dim != 64 && head_dim != 128) return fail(PA_ERR_UNSUPPORTED, "head_dim %d not supported", head_dim);
  if (dtype != PA_F32 && dtype != PA_BF16 && dtype != PA_F16)
    return fail(PA_ERR_UNSUPPORTED, "dtype %d not supported", dtype);
  if (num_tokens < 0 || num_heads < 1 || max_positions < 0)
    return fail(PA_ERR_INVALID, "num_tokens >= 0, num_heads >= 1 and max_positions >= 0 required");
  if (num_tokens == 0) return PA_OK;
  if (!x || !positions || !cos_sin) return fail(PA_ERR_INVALID, "null pointer argument");
  if (!aligned16(x) || (reinterpret_cast<uintptr_t>(positions) & 3u) || (reinterpret_cast<uintptr_t>(cos_sin) & 7u))
    return fail(PA_ERR_INVALID, "x (16), positions (4) or cos_sin (8 bytes) misaligned");
  int* status = status_ptr();
  if (!status) return fail(PA_ERR_CUDA, "no CUDA device / status word unavailable");
  cudaError_t e = pa::launch_apply_rope(x, positions, cos_sin, max_positions, num_tokens, num_heads, head_dim, dtype,
                                        status, static_cast<cudaStream_t>(stream));
  if (e != cudaSuccess) return cuda_fail(e, "apply_rope launch");
  return PA_OK;
}

int pa_copy_blocks(void* k_pool, void* v_pool, const int32_t* pairs, int num_pairs, const pa_pool_desc* pool,
                   void* stream) {
  t_err.clear();
  int rc = check_pool(pool);
  if (rc != PA_OK) return rc;
  if ((rc = reject_int8(pool)) != PA_OK) return rc;
  if (num_pairs < 0) return fail(PA_ERR_INVALID, "num_pairs must be >= 0");
  if (num_pairs == 0) return PA_OK;
  if (!k_pool || !v_pool || !pairs) return fail(PA_ERR_INVALID, "null pointer argument");
  if (!aligned16(k_pool) || !aligned16(v_pool) || (reinterpret_cast<uintptr_t>(pairs) & 7u))
    return fail(PA_ERR_INVALID, "pools must be 16-byte and pairs 8-byte aligned");
  int* status = status_ptr();
  if (!status) return fail(PA_ERR_CUDA, "no CUDA device / status word unavailable");
  const int block_bytes = pool->num_kv_heads * PA_BLOCK_SIZE * pool->head_dim * elem_bytes(pool->dtype);
  pa::CopyArrays arrs{{k_pool, v_pool, nullptr, nullptr}, {block_bytes / 16, block_bytes / 16, 0, 0}};
  cudaError_t e = pa::launch_copy_blocks(arrs, 2, pairs, num_pairs, pool->num_blocks, status,
                                         static_cast<cudaStream_t>(stream));
  if (e != cudaSuccess) return cuda_fail(e, "copy_blocks launch");
  return PA_OK;
}

int pa_copy_blocks_int8(void* k_codes, void* v_codes, float* k_scales, float* v_scales, const int32_t* pairs,
                        int num_pairs, const pa_pool_desc* pool, void* stream) {
  t_err.clear();
  int rc = check_pool(pool);
  if (rc != PA_OK) return rc;
  if (pool->dtype != PA_I8) return fail(PA_ERR_INVALID, "pool dtype must be PA_I8 for an INT8 cache");
  if (num_pairs < 0) return fail(PA_ERR_INVALID, "num_pairs must be >= 0");
  if (num_pairs == 0) return PA_OK;
  if (!k_codes || !v_codes || !k_scales || !v_scales || !pairs) return fail(PA_ERR_INVALID, "null pointer argument");
  if (!aligned16(k_codes) || !aligned16(v_codes) || !aligned16(k_scales) || !aligned16(v_scales) ||
      (reinterpret_cast<uintptr_t>(pairs) & 7u))
    return fail(PA_ERR_INVALID, "codes and scales must be 16-byte and pairs 8-byte aligned");
  int* status = status_ptr();
  if (!status) return fail(PA_ERR_CUDA, "no CUDA device / status word unavailable");
  const int code_bytes = pool->num_kv_heads * PA_BLOCK_SIZE * pool->head_dim;   // one byte per code
  const int scale_bytes = pool->num_kv_heads * PA_BLOCK_SIZE * static_cast<int>(sizeof(float));
  pa::CopyArrays arrs{{k_codes, v_codes, k_scales, v_scales},
                      {code_bytes / 16, code_bytes / 16, scale_bytes / 16, scale_bytes / 16}};
  cudaError_t e = pa::launch_copy_blocks(arrs, 4, pairs, num_pairs, pool->num_blocks, status,
                                         static_cast<cudaStream_t>(stream));
  if (e != cudaSuccess) return cuda_fail(e, "copy_blocks_int8 launch");
  return PA_OK;
}

int pa_device_status(int* status, void* stream) {
  t_err.clear();
  if (!status) return fail(PA_ERR_INVALID, "status pointer is NULL");
  int* dev = status_ptr();
  if (!dev) return fail(PA_ERR_CUDA, "no CUDA device / status word unavailable");
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  int host = 0;
  cudaError_t e = cudaMemcpyAsync(&host, dev, sizeof(int), cudaMemcpyDeviceToHost, st);
  if (e == cudaSuccess) e = cudaMemsetAsync(dev, 0, sizeof(int), st);
  if (e == cudaSuccess) e = cudaStreamSynchronize(st);
  if (e != cudaSuccess) return cuda_fail(e, "device status read");
  *status = host;
  if (host != 0) return fail(PA_ERR_DEVICE, "device status word 0x%x", host);
  return PA_OK;
}

}  // extern "C"
