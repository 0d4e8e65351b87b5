// block_manager.cpp -- host-side bookkeeping of the paged KV pool with a
// prefix cache: block tables, reference counts, copy-on-write, eviction.
//
// The pool of 16-token blocks reached through per-sequence block tables
// ("LLM Inference Server", Optional Bonus Extensions: Paged KV-Cache Block
// Allocator; "LLM Inference Server From Scratch", How it works, 3 Block
// Manager) with the hash-keyed prefix cache of "LLM Inference Server",
// Stage 1 (a common system prompt's KV stored once, reused by later requests,
// hit/miss tracking) and blocks shared across requests ("Mini inference
// engine (KV cache + sampling + quantization)", step 2, stretch).
//
// Policies (deterministic, so every block id is a function of the call
// sequence):
//  * full blocks are keyed by FNV-1a 64 over the little-endian bytes of the
//    parent block's key (0 for the first block) and the 16 token ids; a hit
//    also compares the stored parent key and tokens;
//  * a prompt reuses its cached full blocks from the start until the first
//    miss, then allocates the rest; new full blocks enter the cache at once
//    (a key already present keeps its block);
//  * an append that opens a block allocates one; an append into a last block
//    that another table also holds copies it first (copy-on-write, returned
//    to the caller as a (source, destination) pair for the GPU copy); a block
//    that fills up enters the cache;
//  * freeing releases a sequence's blocks last to first; a cached block whose
//    count reaches zero waits on a least-recently-released list, others go
//    back to the free set;
//  * allocation takes the lowest free id, else evicts the least recently
//    released cached block; when neither exists the call fails with
//    PA_ERR_NO_BLOCKS and changes nothing.
// Not thread-safe: one caller (the scheduler) owns a manager.
#include <cstdint>
#include <cstdio>
#include <new>
#include <set>
#include <unordered_map>
#include <utility>
#include <vector>

#include "pa.h"

namespace pa {
int set_last_error(int code, const char* msg);
}

namespace {

constexpr int B = PA_BLOCK_SIZE;
constexpr uint64_t kFnvOffset = 0xCBF29CE484222325ull;
constexpr uint64_t kFnvPrime = 0x100000001B3ull;

uint64_t fnv_byte(uint64_t h, uint8_t b) { return (h ^ b) * kFnvPrime; }

uint64_t block_key(uint64_t parent, const int32_t* toks) {
  uint64_t h = kFnvOffset;
  for (int i = 0; i < 8; ++i) h = fnv_byte(h, static_cast<uint8_t>(parent >> (8 * i)));
  for (int t = 0; t < B; ++t) {
    const uint32_t u = static_cast<uint32_t>(toks[t]);
    for (int i = 0; i < 4; ++i) h = fnv_byte(h, static_cast<uint8_t>(u >> (8 * i)));
  }
  return h;
}

struct BlockInfo {
  int ref = 0;
  bool keyed = false;     // entered in the cache under `key`
  uint64_t key = 0;
  uint64_t parent = 0;
  int32_t toks[B] = {};
  uint64_t tick = 0;      // release tick while on the LRU list, else 0
};

struct Seq {
  bool live = false;
  std::vector<int32_t> table;
  int len = 0;
  int32_t tail[B] = {};
  int tail_n = 0;
  uint64_t parent = 0;    // key of the last full block
};

int err(int code, const char* msg) { return pa::set_last_error(code, msg); }

}  // namespace

struct pa_block_manager {
  int nb = 0, max_blocks = 0, max_seqs = 0;
  std::vector<BlockInfo> blk;
  std::set<int> free_set;
  std::set<std::pair<uint64_t, int>> lru;
  std::unordered_map<uint64_t, int> cache;
  uint64_t tick = 0;
  std::vector<Seq> seqs;
  pa_bm_stats st{};

  int available() const { return static_cast<int>(free_set.size() + lru.size()); }

  int alloc() {
    int b;
    if (!free_set.empty()) {
      b = *free_set.begin();
      free_set.erase(free_set.begin());
    } else {
      b = lru.begin()->second;   // callers checked availability
      lru.erase(lru.begin());
      BlockInfo& x = blk[b];
      auto it = cache.find(x.key);
      if (x.keyed && it != cache.end() && it->second == b) cache.erase(it);
      x.keyed = false;
      x.tick = 0;
      ++st.evictions;
    }
    blk[b].ref = 1;
    return b;
  }

  uint64_t enter(int b, uint64_t parent, const int32_t* toks) {
    const uint64_t k = block_key(parent, toks);
    if (cache.find(k) == cache.end()) {
      cache.emplace(k, b);
      BlockInfo& x = blk[b];
      x.keyed = true;
      x.key = k;
      x.parent = parent;
      for (int i = 0; i < B; ++i) x.toks[i] = toks[i];
    }
    return k;
  }

  int lookup(uint64_t parent, const int32_t* toks) const {
    auto it = cache.find(block_key(parent, toks));
    if (it == cache.end()) return -1;
    const BlockInfo& x = blk[it->second];
    if (x.parent != parent) return -1;
    for (int i = 0; i < B; ++i)
      if (x.toks[i] != toks[i]) return -1;
    return it->second;
  }

  void take_from_lru(int b) {
    BlockInfo& x = blk[b];
    if (x.ref == 0 && x.tick != 0) {
      lru.erase({x.tick, b});
      x.tick = 0;
    }
  }
};

extern "C" {

pa_block_manager* pa_bm_create(int num_blocks, int max_blocks_per_seq, int max_seqs) {
  if (num_blocks < 1 || max_blocks_per_seq < 1 || max_seqs < 1) {
    err(PA_ERR_INVALID, "num_blocks, max_blocks_per_seq and max_seqs must be >= 1");
    return nullptr;
  }
  pa_block_manager* m = new (std::nothrow) pa_block_manager();
  if (!m) {
    err(PA_ERR_INVALID, "out of host memory");
    return nullptr;
  }
  m->nb = num_blocks;
  m->max_blocks = max_blocks_per_seq;
  m->max_seqs = max_seqs;
  m->blk.resize(num_blocks);
  for (int b = 0; b < num_blocks; ++b) m->free_set.insert(m->free_set.end(), b);
  m->seqs.resize(max_seqs);
  return m;
}

void pa_bm_destroy(pa_block_manager* m) { delete m; }

int pa_bm_add_sequence(pa_block_manager* m, int seq, const int32_t* prompt, int prompt_len, int64_t* slots) {
  if (!m) return err(PA_ERR_INVALID, "null manager");
  if (seq < 0 || seq >= m->max_seqs || m->seqs[seq].live) return err(PA_ERR_INVALID, "bad or live sequence id");
  if (prompt_len < 0 || (prompt_len > 0 && (!prompt || !slots)))
    return err(PA_ERR_INVALID, "bad prompt arguments");
  const int nblocks = (prompt_len + B - 1) / B;
  if (nblocks > m->max_blocks) return err(PA_ERR_INVALID, "prompt longer than the block table");
  const int full = prompt_len / B;
  std::vector<int> hits;
  uint64_t parent = 0;
  for (int i = 0; i < full; ++i) {
    const int b = m->lookup(parent, prompt + i * B);
    if (b < 0) break;
    hits.push_back(b);
    parent = block_key(parent, prompt + i * B);
  }
  int idle_hits = 0;
  for (int b : hits) idle_hits += (m->blk[b].ref == 0) ? 1 : 0;
  if (m->available() - idle_hits < nblocks - static_cast<int>(hits.size()))
    return err(PA_ERR_NO_BLOCKS, "not enough free or evictable blocks for the prompt");
  Seq& s = m->seqs[seq];
  s.table.clear();
  for (int b : hits) {
    m->take_from_lru(b);
    ++m->blk[b].ref;
    s.table.push_back(b);
  }
  m->st.hit_blocks += static_cast<int64_t>(hits.size());
  m->st.miss_blocks += full - static_cast<int64_t>(hits.size());
  for (int i = static_cast<int>(hits.size()); i < nblocks; ++i) {
    const int b = m->alloc();
    s.table.push_back(b);
    if ((i + 1) * B <= prompt_len) parent = m->enter(b, parent, prompt + i * B);
  }
  s.live = true;
  s.len = prompt_len;
  s.tail_n = prompt_len - full * B;
  for (int i = 0; i < s.tail_n; ++i) s.tail[i] = prompt[full * B + i];
  s.parent = parent;
  for (int p = 0; p < prompt_len; ++p) slots[p] = static_cast<int64_t>(s.table[p / B]) * B + p % B;
  return static_cast<int>(hits.size()) * B;
}

int pa_bm_append(pa_block_manager* m, int seq, const int32_t* tokens, int n, int64_t* slots, int32_t* copies,
                 int max_copies, int* num_copies) {
  if (!m) return err(PA_ERR_INVALID, "null manager");
  if (seq < 0 || seq >= m->max_seqs || !m->seqs[seq].live) return err(PA_ERR_INVALID, "sequence is not live");
  if (n < 0 || (n > 0 && (!tokens || !slots)) || !num_copies) return err(PA_ERR_INVALID, "bad append arguments");
  Seq& s = m->seqs[seq];
  *num_copies = 0;
  if (n == 0) return PA_OK;
  if ((static_cast<long long>(s.len) + n + B - 1) / B > m->max_blocks)
    return err(PA_ERR_INVALID, "sequence longer than the block table");
  int opens = 0;
  for (int p = s.len; p < s.len + n; ++p) opens += (p % B == 0) ? 1 : 0;
  const bool cow = (s.len % B != 0) && m->blk[s.table.back()].ref > 1;
  if (cow && (!copies || max_copies < 1)) return err(PA_ERR_INVALID, "a copy-on-write needs room for one pair");
  if (m->available() < opens + (cow ? 1 : 0)) return err(PA_ERR_NO_BLOCKS, "not enough free or evictable blocks");
  for (int i = 0; i < n; ++i) {
    const int p = s.len;
    if (p % B == 0) {
      s.table.push_back(m->alloc());
      s.tail_n = 0;
    } else if (m->blk[s.table.back()].ref > 1) {
      const int src = s.table.back();
      const int dst = m->alloc();
      copies[2 * *num_copies] = src;
      copies[2 * *num_copies + 1] = dst;
      ++*num_copies;
      --m->blk[src].ref;
      s.table.back() = dst;
      ++m->st.cow_copies;
    }
    slots[i] = static_cast<int64_t>(s.table.back()) * B + p % B;
    s.tail[s.tail_n++] = tokens[i];
    s.len = p + 1;
    if (s.len % B == 0) {
      s.parent = m->enter(s.table.back(), s.parent, s.tail);
      s.tail_n = 0;
    }
  }
  return PA_OK;
}

int pa_bm_append_step(pa_block_manager* m, const int32_t* seq_ids, const int32_t* tokens, int n, int64_t* slots,
                      int32_t* copies, int max_copies, int* num_copies) {
  if (!m) return err(PA_ERR_INVALID, "null manager");
  if (n < 0 || (n > 0 && (!seq_ids || !tokens || !slots)) || !num_copies)
    return err(PA_ERR_INVALID, "bad append_step arguments");
  *num_copies = 0;
  // validate and count the blocks the whole step needs before changing anything
  std::unordered_map<int, int> dec;
  std::vector<char> seen(m->max_seqs, 0);
  int need = 0;
  for (int i = 0; i < n; ++i) {
    const int sq = seq_ids[i];
    if (sq < 0 || sq >= m->max_seqs || !m->seqs[sq].live) return err(PA_ERR_INVALID, "sequence is not live");
    if (seen[sq]) return err(PA_ERR_INVALID, "a sequence listed twice");
    seen[sq] = 1;
    const Seq& s = m->seqs[sq];
    if ((s.len + 1 + B - 1) / B > m->max_blocks) return err(PA_ERR_INVALID, "sequence longer than the block table");
    if (s.len % B == 0) {
      ++need;
    } else {
      const int last = s.table.back();
      if (m->blk[last].ref - dec[last] > 1) {
        ++need;
        ++dec[last];
      }
    }
  }
  int pairs = 0;
  for (auto& kv : dec) pairs += kv.second;
  if (pairs > 0 && (!copies || max_copies < pairs)) return err(PA_ERR_INVALID, "copies buffer too small");
  if (m->available() < need) return err(PA_ERR_NO_BLOCKS, "not enough free or evictable blocks");
  for (int i = 0; i < n; ++i) {
    int c = 0;
    const int rc = pa_bm_append(m, seq_ids[i], tokens + i, 1, slots + i, copies ? copies + 2 * *num_copies : nullptr,
                                max_copies - *num_copies, &c);
    if (rc != PA_OK) return rc;   // not reached: every check above passed
    *num_copies += c;
  }
  return PA_OK;
}

int pa_bm_fork(pa_block_manager* m, int parent, int child) {
  if (!m) return err(PA_ERR_INVALID, "null manager");
  if (parent < 0 || parent >= m->max_seqs || !m->seqs[parent].live) return err(PA_ERR_INVALID, "parent not live");
  if (child < 0 || child >= m->max_seqs || m->seqs[child].live) return err(PA_ERR_INVALID, "bad or live child id");
  const Seq& p = m->seqs[parent];
  for (int b : p.table) ++m->blk[b].ref;
  m->seqs[child] = p;
  return PA_OK;
}

int pa_bm_free_sequence(pa_block_manager* m, int seq) {
  if (!m) return err(PA_ERR_INVALID, "null manager");
  if (seq < 0 || seq >= m->max_seqs || !m->seqs[seq].live) return err(PA_ERR_INVALID, "sequence is not live");
  Seq& s = m->seqs[seq];
  for (auto it = s.table.rbegin(); it != s.table.rend(); ++it) {
    BlockInfo& x = m->blk[*it];
    if (--x.ref == 0) {
      auto c = m->cache.find(x.key);
      if (x.keyed && c != m->cache.end() && c->second == *it) {
        x.tick = ++m->tick;
        m->lru.insert({x.tick, *it});
      } else {
        x.keyed = false;
        m->free_set.insert(*it);
      }
    }
  }
  s = Seq();
  return PA_OK;
}

int pa_bm_block_tables(const pa_block_manager* m, const int32_t* seq_ids, int n, int32_t* tables, int max_blocks,
                       int32_t* context_lens) {
  if (!m) return err(PA_ERR_INVALID, "null manager");
  if (n < 0 || (n > 0 && (!seq_ids || !tables || !context_lens)) || max_blocks < 1)
    return err(PA_ERR_INVALID, "bad table arguments");
  for (int i = 0; i < n; ++i) {
    const int sq = seq_ids[i];
    if (sq < 0 || sq >= m->max_seqs || !m->seqs[sq].live) return err(PA_ERR_INVALID, "sequence is not live");
    const Seq& s = m->seqs[sq];
    if (static_cast<int>(s.table.size()) > max_blocks) return err(PA_ERR_INVALID, "table wider than max_blocks");
    for (int j = 0; j < max_blocks; ++j)
      tables[static_cast<size_t>(i) * max_blocks + j] = j < static_cast<int>(s.table.size()) ? s.table[j] : 0;
    context_lens[i] = s.len;
  }
  return PA_OK;
}

int pa_bm_get_stats(const pa_block_manager* m, pa_bm_stats* out) {
  if (!m || !out) return err(PA_ERR_INVALID, "null argument");
  *out = m->st;
  out->free_blocks = static_cast<int32_t>(m->free_set.size());
  out->cached_free_blocks = static_cast<int32_t>(m->lru.size());
  int used = 0;
  for (const BlockInfo& x : m->blk) used += x.ref > 0 ? 1 : 0;
  out->used_blocks = used;
  return PA_OK;
}

}  // extern "C"
