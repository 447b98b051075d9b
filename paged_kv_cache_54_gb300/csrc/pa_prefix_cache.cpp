// Host prefix cache over the block pool: full blocks are keyed by their
// content chained to everything before them, shared through reference
// counts, and kept after their last user leaves until the block is needed
// again (least recently freed first).
//
// Keys.  A full block's key is the 64-bit FNV-1a hash of its parent block's
// key (8 bytes, little-endian; 0 for the first block) followed by its token
// ids (4 bytes each, little-endian).  The cache keeps, for every keyed
// block, the parent key and the token ids, and a lookup only hits when both
// equal the request's: two different prefixes share a block only if their
// parents' 64-bit keys collide.
//
// Free list.  An intrusive doubly linked list over block ids: blocks are
// taken from the front and returned at the back, a hit on a free block
// unlinks it in O(1).  The initial order is the caller's pool order.
#include <cstdint>
#include <cstring>
#include <new>
#include <unordered_map>
#include <vector>

#include "pa.h"

namespace {

constexpr uint64_t kFnvOffset = 14695981039346656037ull;
constexpr uint64_t kFnvPrime = 1099511628211ull;

uint64_t fnv1a_bytes(uint64_t h, const uint8_t *p, size_t n) {
  for (size_t i = 0; i < n; ++i) {
    h ^= p[i];
    h *= kFnvPrime;
  }
  return h;
}

uint64_t block_key(uint64_t parent, const int32_t *tokens, int n) {
  uint8_t buf[8];
  for (int i = 0; i < 8; ++i) buf[i] = static_cast<uint8_t>(parent >> (8 * i));
  uint64_t h = fnv1a_bytes(kFnvOffset, buf, 8);
  for (int t = 0; t < n; ++t) {
    const uint32_t v = static_cast<uint32_t>(tokens[t]);
    for (int i = 0; i < 4; ++i) buf[i] = static_cast<uint8_t>(v >> (8 * i));
    h = fnv1a_bytes(h, buf, 4);
  }
  return h;
}

struct Sequence {
  std::vector<int32_t> table;
  std::vector<int32_t> tokens;
  uint64_t last_key = 0;  // key of the last full block (0 before the first)
};

}  // namespace

struct pa_prefix_cache {
  int32_t num_blocks = 0, block_size = 0;
  std::vector<int32_t> ref;
  // free list
  std::vector<int32_t> prev, next;
  std::vector<uint8_t> in_free;
  int32_t head = -1, tail = -1;
  int64_t free_count = 0;
  // keyed blocks
  std::vector<uint8_t> has_key;
  std::vector<uint64_t> key, parent_key;
  std::vector<int32_t> key_tokens;  // [num_blocks, block_size]
  std::unordered_map<uint64_t, int32_t> block_of;
  std::unordered_map<int64_t, Sequence> seqs;
  int64_t queried_tokens = 0, hit_tokens = 0, evictions = 0;

  void push_back(int32_t b) {
    prev[b] = tail;
    next[b] = -1;
    if (tail >= 0) next[tail] = b; else head = b;
    tail = b;
    in_free[b] = 1;
    ++free_count;
  }
  void unlink(int32_t b) {
    if (prev[b] >= 0) next[prev[b]] = next[b]; else head = next[b];
    if (next[b] >= 0) prev[next[b]] = prev[b]; else tail = prev[b];
    prev[b] = next[b] = -1;
    in_free[b] = 0;
    --free_count;
  }
  // the cached block holding exactly (parent, tokens), or -1
  int32_t lookup(uint64_t parent, const int32_t *tokens) const {
    const uint64_t k = block_key(parent, tokens, block_size);
    auto it = block_of.find(k);
    if (it == block_of.end()) return -1;
    const int32_t b = it->second;
    if (parent_key[b] != parent) return -1;
    if (std::memcmp(&key_tokens[static_cast<size_t>(b) * block_size], tokens,
                    sizeof(int32_t) * block_size) != 0)
      return -1;
    return b;
  }
  int32_t take_fresh() {
    const int32_t b = head;
    unlink(b);
    if (has_key[b]) {
      auto it = block_of.find(key[b]);
      if (it != block_of.end() && it->second == b) block_of.erase(it);
      has_key[b] = 0;
      ++evictions;
    }
    ref[b] = 1;
    return b;
  }
  // key block b as (parent, tokens) unless that content is cached already
  void register_block(int32_t b, uint64_t parent, const int32_t *tokens, uint64_t k) {
    if (block_of.count(k)) return;  // cached in another block (or a colliding key): keep it
    block_of.emplace(k, b);
    has_key[b] = 1;
    key[b] = k;
    parent_key[b] = parent;
    std::memcpy(&key_tokens[static_cast<size_t>(b) * block_size], tokens, sizeof(int32_t) * block_size);
  }
};

extern "C" {

PA_API pa_prefix_cache *pa_prefix_cache_create(int32_t num_blocks, int32_t block_size,
                                               const int32_t *pool_order) {
  if (num_blocks <= 0 || block_size <= 0) return nullptr;
  pa_prefix_cache *c = new (std::nothrow) pa_prefix_cache();
  if (c == nullptr) return nullptr;
  try {
    c->num_blocks = num_blocks;
    c->block_size = block_size;
    c->ref.assign(num_blocks, 0);
    c->prev.assign(num_blocks, -1);
    c->next.assign(num_blocks, -1);
    c->in_free.assign(num_blocks, 0);
    c->has_key.assign(num_blocks, 0);
    c->key.assign(num_blocks, 0);
    c->parent_key.assign(num_blocks, 0);
    c->key_tokens.assign(static_cast<size_t>(num_blocks) * block_size, 0);
    for (int32_t i = 0; i < num_blocks; ++i) {
      const int32_t b = pool_order ? pool_order[i] : i;
      if (b < 0 || b >= num_blocks || c->in_free[b]) {  // not a permutation
        delete c;
        return nullptr;
      }
      c->push_back(b);
    }
  } catch (...) {
    delete c;
    return nullptr;
  }
  return c;
}

PA_API void pa_prefix_cache_destroy(pa_prefix_cache *c) { delete c; }

PA_API pa_status pa_prefix_cache_add_sequence(pa_prefix_cache *c, int64_t seq_id, const int32_t *tokens,
                                              int32_t num_tokens, int32_t *num_cached_tokens) {
  if (c == nullptr || num_tokens < 0 || (num_tokens > 0 && tokens == nullptr)) return PA_ERR_INVALID;
  if (c->seqs.count(seq_id)) return PA_ERR_INVALID;
  const int bs = c->block_size;
  const int32_t nfull = num_tokens / bs;
  const int32_t nblocks = (num_tokens + bs - 1) / bs;
  // longest run of cached full blocks from the start
  std::vector<int32_t> hits;
  std::vector<uint64_t> keys;
  uint64_t parent = 0;
  try {
    hits.reserve(nfull);
    keys.reserve(nfull);
    for (int32_t j = 0; j < nfull; ++j) {
      const int32_t *tk = tokens + static_cast<size_t>(j) * bs;
      keys.push_back(block_key(parent, tk, bs));
      if (static_cast<int32_t>(hits.size()) == j) {
        const int32_t b = c->lookup(parent, tk);
        if (b >= 0) hits.push_back(b);
      }
      parent = keys.back();
    }
    int64_t free_hits = 0;
    for (int32_t b : hits) free_hits += c->ref[b] == 0;
    const int64_t need = static_cast<int64_t>(nblocks - static_cast<int32_t>(hits.size())) + free_hits;
    if (need > c->free_count) return PA_ERR_OUT_OF_BLOCKS;
    Sequence s;
    s.table.reserve(nblocks);
    s.tokens.assign(tokens, tokens + num_tokens);
    for (int32_t b : hits) {
      if (c->ref[b] == 0) c->unlink(b);
      ++c->ref[b];
      s.table.push_back(b);
    }
    for (int32_t j = static_cast<int32_t>(hits.size()); j < nblocks; ++j) {
      const int32_t b = c->take_fresh();
      s.table.push_back(b);
      if (j < nfull)
        c->register_block(b, j ? keys[j - 1] : 0, tokens + static_cast<size_t>(j) * bs, keys[j]);
    }
    s.last_key = nfull ? keys[nfull - 1] : 0;
    c->seqs.emplace(seq_id, std::move(s));
  } catch (...) {
    return PA_ERR_INVALID;  // out of host memory
  }
  c->queried_tokens += num_tokens;
  c->hit_tokens += static_cast<int64_t>(hits.size()) * bs;
  if (num_cached_tokens) *num_cached_tokens = static_cast<int32_t>(hits.size()) * bs;
  return PA_OK;
}

PA_API pa_status pa_prefix_cache_append_token(pa_prefix_cache *c, int64_t seq_id, int32_t token,
                                              int64_t *slot) {
  if (c == nullptr) return PA_ERR_INVALID;
  auto it = c->seqs.find(seq_id);
  if (it == c->seqs.end()) return PA_ERR_INVALID;
  Sequence &s = it->second;
  const int bs = c->block_size;
  const int64_t pos = static_cast<int64_t>(s.tokens.size());
  try {
    if (pos % bs == 0) {
      if (c->free_count == 0) return PA_ERR_OUT_OF_BLOCKS;
      s.table.push_back(c->take_fresh());
    }
    s.tokens.push_back(token);
  } catch (...) {
    return PA_ERR_INVALID;
  }
  if (s.tokens.size() % bs == 0) {  // the last block just filled: key it
    const size_t j = s.tokens.size() / bs - 1;
    const int32_t *tk = s.tokens.data() + j * bs;
    const uint64_t k = block_key(s.last_key, tk, bs);
    c->register_block(s.table[j], s.last_key, tk, k);
    s.last_key = k;
  }
  if (slot) *slot = static_cast<int64_t>(s.table[pos / bs]) * bs + pos % bs;
  return PA_OK;
}

PA_API pa_status pa_prefix_cache_free_sequence(pa_prefix_cache *c, int64_t seq_id) {
  if (c == nullptr) return PA_ERR_INVALID;
  auto it = c->seqs.find(seq_id);
  if (it == c->seqs.end()) return PA_ERR_INVALID;
  const std::vector<int32_t> &t = it->second.table;
  for (auto b = t.rbegin(); b != t.rend(); ++b)  // last block first: tails are evicted first
    if (--c->ref[*b] == 0) c->push_back(*b);
  c->seqs.erase(it);
  return PA_OK;
}

PA_API int32_t pa_prefix_cache_block_table(const pa_prefix_cache *c, int64_t seq_id, int32_t *table,
                                           int32_t capacity, int32_t *num_tokens) {
  if (c == nullptr) return -1;
  auto it = c->seqs.find(seq_id);
  if (it == c->seqs.end()) return -1;
  const std::vector<int32_t> &t = it->second.table;
  if (num_tokens) *num_tokens = static_cast<int32_t>(it->second.tokens.size());
  const int32_t n = static_cast<int32_t>(t.size());
  if (table != nullptr)
    for (int32_t i = 0; i < n && i < capacity; ++i) table[i] = t[i];
  return n;
}

PA_API pa_status pa_prefix_cache_block_tables(const pa_prefix_cache *c, const int64_t *seq_ids,
                                              int32_t num_seqs, int32_t *tables, int32_t width,
                                              int32_t *seq_lens) {
  if (c == nullptr || num_seqs < 0 || width <= 0 || (num_seqs > 0 && (!seq_ids || !tables)))
    return PA_ERR_INVALID;
  for (int32_t i = 0; i < num_seqs; ++i) {
    auto it = c->seqs.find(seq_ids[i]);
    if (it == c->seqs.end()) return PA_ERR_INVALID;
    if (static_cast<int32_t>(it->second.table.size()) > width) return PA_ERR_INVALID;
  }
  for (int32_t i = 0; i < num_seqs; ++i) {
    const Sequence &s = c->seqs.find(seq_ids[i])->second;
    int32_t *row = tables + static_cast<size_t>(i) * width;
    const int32_t n = static_cast<int32_t>(s.table.size());
    for (int32_t j = 0; j < width; ++j) row[j] = j < n ? s.table[j] : 0;
    if (seq_lens) seq_lens[i] = static_cast<int32_t>(s.tokens.size());
  }
  return PA_OK;
}

PA_API pa_status pa_prefix_cache_get_stats(const pa_prefix_cache *c, pa_prefix_cache_stats *out) {
  if (c == nullptr || out == nullptr) return PA_ERR_INVALID;
  int64_t cached_free = 0;
  for (int32_t b = c->head; b >= 0; b = c->next[b]) cached_free += c->has_key[b];
  out->free_blocks = c->free_count;
  out->cached_free_blocks = cached_free;
  out->used_blocks = c->num_blocks - c->free_count;
  out->cached_blocks = static_cast<int64_t>(c->block_of.size());
  out->queried_tokens = c->queried_tokens;
  out->hit_tokens = c->hit_tokens;
  out->evictions = c->evictions;
  return PA_OK;
}

PA_API int32_t pa_prefix_cache_free_order(const pa_prefix_cache *c, int32_t *out, int32_t capacity) {
  if (c == nullptr) return -1;
  int32_t n = 0;
  for (int32_t b = c->head; b >= 0; b = c->next[b], ++n)
    if (out != nullptr && n < capacity) out[n] = b;
  return n;
}

PA_API int32_t pa_prefix_cache_ref_count(const pa_prefix_cache *c, int32_t block) {
  if (c == nullptr || block < 0 || block >= c->num_blocks) return -1;
  return c->ref[block];
}

}  // extern "C"
