// block_manager.cpp -- the host side of the paged KV cache: physical blocks,
// reference counts, copy-on-write and the prefix hash chain.
//
// "KV cache, prefill và decode", section 05 ("Block table", "Chia sẻ block và
// copy-on-write", "Prefix caching"): the cache is cut into fixed-size blocks;
// a sequence gets a new block only when its last one is full; every physical
// block has a reference count; sequences forked from one prompt (parallel
// sampling) share its blocks, and a shared block is copied before a sequence
// writes into it; a full block is identified by a hash of its own tokens and
// of its parent block's hash (the whole prefix up to it), and a new request
// that finds the hash reuses the block (reference count + 1) and skips that
// part of the prefill.  "Inference part 1", section "Prefix caching": the
// lookup walks the prompt's blocks from the start and stops at the first
// miss.  "Efficient Inference", section on paged attention: a finished
// request's blocks return to the free pool.  Cached blocks nobody holds are
// evicted least recently used first when the pool runs dry (the pages name
// LRU eviction for RadixAttention's cached prefixes).
//
// Policy details the pages leave open (each stated where it is used):
//   * free blocks are reused last-freed first (a stack);
//   * a block becomes cached the moment it is full; an identical full block
//     computed by another sequence is not merged (the first one stays in the
//     table);
//   * eviction takes the cached, unreferenced block with the oldest last use,
//     ties by lower block id; a lookup hit or a release counts as a use;
//   * the block hash is 64-bit FNV-1a over the parent hash (8 bytes, little
//     endian; 0 for the first block) followed by the block's token ids (4
//     bytes each, little endian).
#include <cstdint>
#include <cstring>
#include <map>
#include <new>
#include <set>
#include <unordered_map>
#include <utility>
#include <vector>

#include "../../include/pkv.h"

namespace pkv {
namespace {

constexpr uint64_t kFnvOffset = 14695981039346656037ull;
constexpr uint64_t kFnvPrime = 1099511628211ull;

uint64_t fnv1a(uint64_t h, const void *data, size_t n) {
  const unsigned char *p = static_cast<const unsigned char *>(data);
  for (size_t i = 0; i < n; ++i) {
    h ^= p[i];
    h *= kFnvPrime;
  }
  return h;
}

uint64_t block_hash(uint64_t parent, const int32_t *tokens, int n) {
  unsigned char buf[8];
  for (int i = 0; i < 8; ++i) buf[i] = static_cast<unsigned char>(parent >> (8 * i));
  uint64_t h = fnv1a(kFnvOffset, buf, 8);
  for (int t = 0; t < n; ++t) {
    const uint32_t v = static_cast<uint32_t>(tokens[t]);
    unsigned char w[4] = {static_cast<unsigned char>(v), static_cast<unsigned char>(v >> 8),
                          static_cast<unsigned char>(v >> 16), static_cast<unsigned char>(v >> 24)};
    h = fnv1a(h, w, 4);
  }
  return h;
}

struct Block {
  int32_t ref = 0;
  bool cached = false;  // full, and registered under `hash`
  uint64_t hash = 0;
  int64_t last_use = 0;
};

struct Sequence {
  std::vector<int32_t> blocks;
  std::vector<int32_t> tokens;
};

}  // namespace
}  // namespace pkv

struct pkv_block_manager {
  int64_t num_blocks = 0;
  int block_size = 0;
  int64_t clock = 0;
  std::vector<pkv::Block> blocks;
  std::vector<int32_t> free_stack;                       // unreferenced, not cached
  std::set<std::pair<int64_t, int32_t>> evictable;       // (last use, id): cached, unreferenced
  std::unordered_map<uint64_t, int32_t> by_hash;         // cached full blocks
  std::map<int64_t, pkv::Sequence> seqs;

  int32_t allocate() {
    if (!free_stack.empty()) {
      const int32_t b = free_stack.back();
      free_stack.pop_back();
      blocks[b] = pkv::Block{};
      blocks[b].ref = 1;
      blocks[b].last_use = ++clock;
      return b;
    }
    if (evictable.empty()) return -1;
    const int32_t b = evictable.begin()->second;
    evictable.erase(evictable.begin());
    by_hash.erase(blocks[b].hash);
    blocks[b] = pkv::Block{};
    blocks[b].ref = 1;
    blocks[b].last_use = ++clock;
    return b;
  }

  void retain(int32_t b) {
    if (blocks[b].ref == 0 && blocks[b].cached) evictable.erase({blocks[b].last_use, b});
    ++blocks[b].ref;
    blocks[b].last_use = ++clock;
  }

  void release(int32_t b) {
    if (--blocks[b].ref > 0) return;
    blocks[b].last_use = ++clock;
    if (blocks[b].cached)
      evictable.insert({blocks[b].last_use, b});
    else
      free_stack.push_back(b);
  }

  // Register sequence s's block i if it has just become full.
  void seal(pkv::Sequence &s, size_t i) {
    const int32_t b = s.blocks[i];
    if (blocks[b].cached) return;
    const uint64_t parent = i == 0 ? 0ull : blocks[s.blocks[i - 1]].hash;
    const uint64_t h = pkv::block_hash(parent, s.tokens.data() + i * block_size, block_size);
    blocks[b].hash = h;
    if (by_hash.count(h)) return;  // an identical block is cached already: not merged
    blocks[b].cached = true;
    by_hash[h] = b;
  }
};

using pkv_bm = pkv_block_manager;

namespace {
// The manager's vectors, maps and sets allocate host memory and may throw
// std::bad_alloc; no exception crosses the C boundary.
template <typename F> pkv_status guarded(F &&body) {
  try {
    return body();
  } catch (...) {
    return PKV_ERR_HOST_MEMORY;
  }
}
}  // namespace

extern "C" {

pkv_block_manager *pkv_bm_create(int64_t num_blocks, int block_size) {
  if (num_blocks < 1 || num_blocks > (int64_t(1) << 31) - 1 || block_size < 1) return nullptr;
  pkv_bm *m = new (std::nothrow) pkv_bm;
  if (!m) return nullptr;
  try {
    m->num_blocks = num_blocks;
    m->block_size = block_size;
    m->blocks.resize(static_cast<size_t>(num_blocks));
    m->free_stack.reserve(static_cast<size_t>(num_blocks));
  } catch (...) {
    delete m;
    return nullptr;
  }
  // within the reserved capacity: no allocation
  for (int64_t b = num_blocks - 1; b >= 0; --b) m->free_stack.push_back(static_cast<int32_t>(b));
  return m;
}

void pkv_bm_destroy(pkv_block_manager *m) { delete m; }

pkv_status pkv_bm_stats(const pkv_block_manager *m, int64_t *free_blocks, int64_t *cached_blocks,
                        int64_t *num_sequences) {
  if (!m) return PKV_ERR_INVALID_ARG;
  if (free_blocks) *free_blocks = static_cast<int64_t>(m->free_stack.size());
  if (cached_blocks) *cached_blocks = static_cast<int64_t>(m->by_hash.size());
  if (num_sequences) *num_sequences = static_cast<int64_t>(m->seqs.size());
  return PKV_OK;
}

pkv_status pkv_bm_block_info(const pkv_block_manager *m, int32_t block, int32_t *ref,
                             int32_t *cached, uint64_t *hash) {
  if (!m || block < 0 || block >= m->num_blocks) return PKV_ERR_INVALID_ARG;
  const pkv::Block &b = m->blocks[block];
  if (ref) *ref = b.ref;
  if (cached) *cached = b.cached ? 1 : 0;
  if (hash) *hash = b.hash;
  return PKV_OK;
}

pkv_status pkv_bm_append(pkv_block_manager *m, int64_t seq_id, const int32_t *tokens, int n,
                         int64_t *slots, int32_t *cow_src, int32_t *cow_dst, int *num_cow);

pkv_status pkv_bm_add_sequence(pkv_block_manager *m, int64_t seq_id, const int32_t *tokens, int n,
                               int use_prefix_cache, int *cached_tokens, int64_t *slots) {
  if (!m || n < 0 || (n > 0 && !tokens) || m->seqs.count(seq_id)) return PKV_ERR_INVALID_ARG;
  return guarded([&]() -> pkv_status {
    const int bs = m->block_size;
    // Prefix lookup, taking nothing yet: walk the prompt's full blocks from the
    // start and stop at the first miss.
    std::vector<int32_t> hits;
    if (use_prefix_cache) {
      uint64_t parent = 0;
      for (int i = 0; static_cast<int64_t>(i + 1) * bs <= n; ++i) {
        const uint64_t h = pkv::block_hash(parent, tokens + static_cast<int64_t>(i) * bs, bs);
        const auto it = m->by_hash.find(h);
        if (it == m->by_hash.end()) break;
        hits.push_back(it->second);
        parent = h;
      }
    }
    const int cached = static_cast<int>(hits.size()) * bs;
    // Capacity for the rest of the prompt, checked before anything changes; a
    // hit that nobody holds stops being evictable once it is taken.
    int64_t avail = static_cast<int64_t>(m->free_stack.size() + m->evictable.size());
    for (int32_t b : hits)
      if (m->blocks[b].ref == 0) --avail;
    if ((static_cast<int64_t>(n - cached) + bs - 1) / bs > avail) return PKV_ERR_WORKSPACE;
    pkv::Sequence &s = m->seqs[seq_id];
    for (int32_t b : hits) {
      m->retain(b);
      s.blocks.push_back(b);
    }
    s.tokens.assign(tokens, tokens + cached);
    if (cached_tokens) *cached_tokens = cached;
    int num_cow = 0;
    return pkv_bm_append(m, seq_id, tokens + cached, n - cached, slots, nullptr, nullptr, &num_cow);
  });
}

pkv_status pkv_bm_append(pkv_block_manager *m, int64_t seq_id, const int32_t *tokens, int n,
                         int64_t *slots, int32_t *cow_src, int32_t *cow_dst, int *num_cow) {
  if (!m || n < 0 || (n > 0 && !tokens)) return PKV_ERR_INVALID_ARG;
  const auto it = m->seqs.find(seq_id);
  if (it == m->seqs.end()) return PKV_ERR_INVALID_ARG;
  return guarded([&]() -> pkv_status {
    pkv::Sequence &s = it->second;
    const int bs = m->block_size;
    // Blocks this call needs: new ones, plus one copy if the last block is
    // shared and will be written.  Checked first, so a call that cannot be
    // served changes nothing.
    const size_t len = s.tokens.size();
    const size_t have = s.blocks.size();
    const size_t need = (len + static_cast<size_t>(n) + bs - 1) / bs;
    int64_t want = static_cast<int64_t>(need > have ? need - have : 0);
    const bool cow = n > 0 && len % bs != 0 && m->blocks[s.blocks.back()].ref > 1;
    if (cow) ++want;
    if (want > static_cast<int64_t>(m->free_stack.size() + m->evictable.size()))
      return PKV_ERR_WORKSPACE;
    // the sequence's own growth, reserved before anything changes
    s.blocks.reserve(need);
    s.tokens.reserve(len + static_cast<size_t>(n));
    int ncow = 0;
    if (cow) {
      // copy-on-write: the sequence gets its own copy of the shared partial
      // block before writing into it
      const int32_t src = s.blocks.back();
      const int32_t dst = m->allocate();
      m->release(src);
      s.blocks.back() = dst;
      if (cow_src) cow_src[0] = src;
      if (cow_dst) cow_dst[0] = dst;
      ncow = 1;
    }
    for (int t = 0; t < n; ++t) {
      const size_t pos = s.tokens.size();
      if (pos % bs == 0) s.blocks.push_back(m->allocate());
      const int32_t b = s.blocks[pos / bs];
      if (slots) slots[t] = static_cast<int64_t>(b) * bs + static_cast<int64_t>(pos % bs);
      s.tokens.push_back(tokens[t]);
      if ((pos + 1) % bs == 0) m->seal(s, pos / bs);
    }
    if (num_cow) *num_cow = ncow;
    return PKV_OK;
  });
}

pkv_status pkv_bm_fork(pkv_block_manager *m, int64_t parent, int64_t child) {
  if (!m || m->seqs.count(child)) return PKV_ERR_INVALID_ARG;
  const auto it = m->seqs.find(parent);
  if (it == m->seqs.end()) return PKV_ERR_INVALID_ARG;
  return guarded([&]() -> pkv_status {
    pkv::Sequence copy = it->second;  // allocated before any count changes
    auto &slot = m->seqs[child];
    for (int32_t b : copy.blocks) m->retain(b);
    slot = std::move(copy);
    return PKV_OK;
  });
}

pkv_status pkv_bm_free(pkv_block_manager *m, int64_t seq_id) {
  if (!m) return PKV_ERR_INVALID_ARG;
  const auto it = m->seqs.find(seq_id);
  if (it == m->seqs.end()) return PKV_ERR_INVALID_ARG;
  return guarded([&]() -> pkv_status {
    for (int32_t b : it->second.blocks) m->release(b);
    m->seqs.erase(it);
    return PKV_OK;
  });
}

pkv_status pkv_bm_sequence(const pkv_block_manager *m, int64_t seq_id, int32_t *blocks,
                           int max_blocks, int *num_blocks, int *num_tokens) {
  if (!m) return PKV_ERR_INVALID_ARG;
  const auto it = m->seqs.find(seq_id);
  if (it == m->seqs.end()) return PKV_ERR_INVALID_ARG;
  const pkv::Sequence &s = it->second;
  if (num_blocks) *num_blocks = static_cast<int>(s.blocks.size());
  if (num_tokens) *num_tokens = static_cast<int>(s.tokens.size());
  if (blocks) {
    if (static_cast<int>(s.blocks.size()) > max_blocks) return PKV_ERR_INVALID_ARG;
    for (size_t i = 0; i < s.blocks.size(); ++i) blocks[i] = s.blocks[i];
  }
  return PKV_OK;
}

pkv_status pkv_bm_block_table(const pkv_block_manager *m, const int64_t *seq_ids, int num_seqs,
                              int32_t *table, int max_blocks_per_seq, int32_t *context_lens) {
  if (!m || num_seqs < 0 || (num_seqs > 0 && (!seq_ids || !table || !context_lens)) ||
      max_blocks_per_seq < 1)
    return PKV_ERR_INVALID_ARG;
  for (int i = 0; i < num_seqs; ++i) {
    const auto it = m->seqs.find(seq_ids[i]);
    if (it == m->seqs.end()) return PKV_ERR_INVALID_ARG;
    const pkv::Sequence &s = it->second;
    if (static_cast<int>(s.blocks.size()) > max_blocks_per_seq) return PKV_ERR_INVALID_ARG;
    int32_t *row = table + static_cast<int64_t>(i) * max_blocks_per_seq;
    for (int j = 0; j < max_blocks_per_seq; ++j)
      row[j] = j < static_cast<int>(s.blocks.size()) ? s.blocks[j] : -1;
    context_lens[i] = static_cast<int32_t>(s.tokens.size());
  }
  return PKV_OK;
}

uint64_t pkv_bm_hash(uint64_t parent_hash, const int32_t *tokens, int n) {
  return pkv::block_hash(parent_hash, tokens, n);
}

}  // extern "C"
