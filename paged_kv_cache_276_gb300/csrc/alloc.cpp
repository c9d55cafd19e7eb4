// Host block allocator behind the pkv_alloc_* / pkv_seq_* C ABI.
//
// A pool of interchangeable fixed-size blocks, one block table per sequence
// (logical order kept, physical placement free), allocation on growth, return
// to the pool on finish (x321.org "The serving bottleneck is not just FLOPs",
// section "PagedAttention borrows an operating-system trick") and
// reference-counted sharing with copy-on-write (praveentn.live "PagedAttention
// KV-cache constraint", section "What the change bought"); under memory
// pressure a sequence's blocks can be swapped out to host memory and back
// (same page, "What it cost").
//
// Full blocks can also be content-addressed (prefix caching): a block filled
// through pkv_seq_append_tokens is registered under a key of its whole token
// prefix, and a later sequence whose tokens match that prefix exactly reuses
// the block instead of storing the same keys and values again (praveentn.live
// "PagedAttention KV-cache constraint", "What the change bought": blocks with
// an identical prefix are shared).  The key of block j is a 128-bit chained
// hash of block j-1's key and block j's token ids (FNV-1a 64 and a splitmix64
// stream), and a hit also compares the block's own token ids, so a false
// match needs a 128-bit collision of the parent key.  A registered block whose
// last owner goes away stays cached as "evictable" (least recently released
// first); taking a block uses the free stack first and evicts only when it is
// empty.
//
// Every mutating call validates first and mutates last, so a failing call
// leaves the state unchanged.
#include <cstdint>
#include <algorithm>
#include <cstring>
#include <list>
#include <new>
#include <unordered_map>
#include <vector>

#include "pkv.h"

namespace {

// Content key of a full block: its whole token prefix, hashed.
struct Key {
  uint64_t h0 = 0, h1 = 0;
  bool operator==(const Key &o) const { return h0 == o.h0 && h1 == o.h1; }
};
struct KeyHash {
  size_t operator()(const Key &k) const { return static_cast<size_t>(k.h0 ^ (k.h1 * 0x9E3779B97F4A7C15ull)); }
};

uint64_t splitmix64(uint64_t x) {  // Steele, Lea and Flood's SplitMix64 finaliser
  x += 0x9E3779B97F4A7C15ull;
  x = (x ^ (x >> 30)) * 0xBF58476D1CE4E5B9ull;
  x = (x ^ (x >> 27)) * 0x94D049BB133111EBull;
  return x ^ (x >> 31);
}

// Key of a block = f(parent key, its token ids).
Key chain_key(const Key &parent, const int32_t *tokens, int n) {
  uint64_t a = 0xCBF29CE484222325ull;  // FNV-1a 64 offset basis
  auto fnv = [&](uint64_t w) {
    for (int i = 0; i < 8; ++i) {
      a ^= (w >> (8 * i)) & 0xFFu;
      a *= 0x100000001B3ull;  // FNV-1a 64 prime
    }
  };
  uint64_t b = splitmix64(parent.h1 ^ 0x5851F42D4C957F2Dull);
  fnv(parent.h0);
  fnv(parent.h1);
  b = splitmix64(b ^ parent.h0);
  for (int i = 0; i < n; ++i) {
    const uint64_t w = static_cast<uint32_t>(tokens[i]);
    fnv(w);
    b = splitmix64(b ^ w);
  }
  return Key{a, b};
}

struct Sequence {
  std::vector<int32_t> blocks;  // logical -> physical
  int64_t len = 0;              // tokens stored
  bool swapped = false;         // blocks released to the pool, contents held by the caller
  bool tracked = true;          // every token came with its id (prefix caching possible)
  Key last_key;                 // key of the last full block (tracked only; the empty prefix: {0, 0})
  std::vector<int32_t> tail;    // token ids of the last, partial block (tracked only)
};

}  // namespace

struct pkv_alloc {
  int32_t num_blocks = 0;
  int32_t block_size = 0;
  std::vector<int32_t> free_stack;  // top = back()
  std::vector<int32_t> refcount;
  std::unordered_map<int64_t, Sequence> seqs;
  // prefix cache
  std::unordered_map<Key, int32_t, KeyHash> cache;  // key -> registered block
  std::vector<Key> block_key;                        // per block, valid while registered
  std::vector<uint8_t> registered;
  std::vector<std::vector<int32_t>> block_tokens;    // per registered block: its token ids
  std::list<int32_t> evictable;                      // registered blocks nobody holds, oldest first
  std::vector<std::list<int32_t>::iterator> evict_pos;

  int64_t available() const { return static_cast<int64_t>(free_stack.size() + evictable.size()); }
  // A block for new data: the free stack first, else the oldest evictable one
  // (dropped from the cache).  The caller has checked available() > 0.
  int32_t take_block() {
    int32_t b;
    if (!free_stack.empty()) {
      b = free_stack.back();
      free_stack.pop_back();
    } else {
      b = evictable.front();
      evictable.pop_front();
      unregister(b);
    }
    refcount[b] = 1;
    return b;
  }
  void release_block(int32_t b) {
    if (--refcount[b] > 0) return;
    if (registered[b]) evict_pos[b] = evictable.insert(evictable.end(), b);
    else free_stack.push_back(b);
  }
  void unregister(int32_t b) {
    cache.erase(block_key[b]);
    registered[b] = 0;
    block_tokens[b].clear();
  }
  // Register a full block under `key` unless that key already names a block.
  void register_block(int32_t b, const Key &key, const int32_t *tokens) {
    if (registered[b] || cache.count(key)) return;
    cache.emplace(key, b);
    block_key[b] = key;
    registered[b] = 1;
    block_tokens[b].assign(tokens, tokens + block_size);
  }
  // The registered block holding exactly `tokens` after the prefix `parent`, or -1.
  int32_t lookup(const Key &key, const int32_t *tokens) const {
    auto it = cache.find(key);
    if (it == cache.end()) return -1;
    const std::vector<int32_t> &t = block_tokens[it->second];
    return std::memcmp(t.data(), tokens, block_size * sizeof(int32_t)) == 0 ? it->second : -1;
  }

  Sequence *find(int64_t id) {
    auto it = seqs.find(id);
    return it == seqs.end() ? nullptr : &it->second;
  }
  const Sequence *find(int64_t id) const {
    auto it = seqs.find(id);
    return it == seqs.end() ? nullptr : &it->second;
  }
  int64_t blocks_for(int64_t tokens) const { return (tokens + block_size - 1) / block_size; }
};

extern "C" {

int pkv_alloc_create(int num_blocks, int block_size, pkv_alloc **out) {
  if (!out || num_blocks < 0 || block_size < 1) return PKV_ERR_ARG;
  pkv_alloc *a = new (std::nothrow) pkv_alloc;
  if (!a) return PKV_ERR_OOM;
  a->num_blocks = num_blocks;
  a->block_size = block_size;
  a->free_stack.resize(num_blocks);
  for (int i = 0; i < num_blocks; ++i) a->free_stack[i] = num_blocks - 1 - i;
  a->refcount.assign(num_blocks, 0);
  a->block_key.assign(num_blocks, Key{});
  a->registered.assign(num_blocks, 0);
  a->block_tokens.assign(num_blocks, {});
  a->evict_pos.resize(num_blocks);
  *out = a;
  return PKV_OK;
}

void pkv_alloc_destroy(pkv_alloc *a) { delete a; }

int pkv_seq_add(pkv_alloc *a, int64_t seq_id) {
  if (!a || a->find(seq_id)) return PKV_ERR_ARG;
  a->seqs.emplace(seq_id, Sequence{});
  return PKV_OK;
}

int pkv_seq_append(pkv_alloc *a, int64_t seq_id, int n_tokens, int64_t *slots_out) {
  if (!a || n_tokens < 0) return PKV_ERR_ARG;
  Sequence *s = a->find(seq_id);
  if (!s || s->swapped) return PKV_ERR_ARG;
  if (n_tokens == 0) return PKV_OK;
  if (!slots_out) return PKV_ERR_ARG;
  const int64_t bs = a->block_size;
  if (s->len % bs != 0) {
    const int32_t last = s->blocks.back();
    if (a->refcount[last] > 1) return PKV_ERR_SHARED;
  }
  const int64_t new_len = s->len + n_tokens;
  const int64_t need = a->blocks_for(new_len) - static_cast<int64_t>(s->blocks.size());
  if (need > a->available()) return PKV_ERR_OOM;
  for (int64_t i = 0; i < need; ++i) s->blocks.push_back(a->take_block());
  for (int64_t pos = s->len, i = 0; pos < new_len; ++pos, ++i)
    slots_out[i] = static_cast<int64_t>(s->blocks[pos / bs]) * bs + pos % bs;
  s->len = new_len;
  s->tracked = false;  // tokens without ids: no prefix caching from here on
  s->tail.clear();
  return PKV_OK;
}

int pkv_seq_append_tokens(pkv_alloc *a, int64_t seq_id, const int32_t *token_ids, int n_tokens,
                          int64_t *slots_out, int *cached_out) {
  if (!a || n_tokens < 0 || !cached_out) return PKV_ERR_ARG;
  Sequence *s = a->find(seq_id);
  if (!s || s->swapped) return PKV_ERR_ARG;
  *cached_out = 0;
  if (n_tokens == 0) return PKV_OK;
  if (!token_ids || !slots_out) return PKV_ERR_ARG;
  const int64_t bs = a->block_size;
  const int64_t len0 = s->len, len1 = len0 + n_tokens;
  if (len0 % bs != 0 && a->refcount[s->blocks.back()] > 1) return PKV_ERR_SHARED;

  // ---- plan: which full blocks of this call are already cached (resolved
  // before anything is taken, so no eviction here can undo a hit)
  const int64_t head = std::min<int64_t>(n_tokens, len0 % bs ? bs - len0 % bs : 0);  // fills the open block
  const int64_t nfull = (n_tokens - head) / bs;                                      // whole blocks after it
  const int64_t tail = n_tokens - head - nfull * bs;
  std::vector<int32_t> hit(nfull, -1);
  std::vector<Key> keys(nfull);
  Key parent = s->last_key;
  Key head_key{};
  const bool head_closes = head > 0 && (len0 + head) % bs == 0;
  if (s->tracked && head_closes) {
    std::vector<int32_t> t(s->tail);
    t.insert(t.end(), token_ids, token_ids + head);
    head_key = chain_key(parent, t.data(), static_cast<int>(bs));
    parent = head_key;
  }
  int64_t revive = 0, fresh = tail > 0 ? 1 : 0;
  for (int64_t j = 0; j < nfull; ++j) {
    const int32_t *t = token_ids + head + j * bs;
    if (s->tracked) {
      keys[j] = chain_key(parent, t, static_cast<int>(bs));
      parent = keys[j];
      hit[j] = a->lookup(keys[j], t);
    }
    if (hit[j] < 0) ++fresh;
    else if (a->refcount[hit[j]] == 0) ++revive;
  }
  if (fresh > a->available() - revive) return PKV_ERR_OOM;

  // ---- apply
  for (int64_t j = 0; j < nfull; ++j) {  // hold the hits first
    const int32_t b = hit[j];
    if (b < 0) continue;
    if (a->refcount[b] == 0) a->evictable.erase(a->evict_pos[b]);
    a->refcount[b] += 1;
  }
  int64_t pos = len0;
  int64_t *slot = slots_out;
  int cached = 0;
  for (int64_t i = 0; i < head; ++i, ++pos) *slot++ = static_cast<int64_t>(s->blocks[pos / bs]) * bs + pos % bs;
  if (s->tracked && head_closes) {
    std::vector<int32_t> t(s->tail);
    t.insert(t.end(), token_ids, token_ids + head);
    a->register_block(s->blocks.back(), head_key, t.data());
  }
  for (int64_t j = 0; j < nfull; ++j) {
    const int32_t *t = token_ids + head + j * bs;
    if (hit[j] >= 0) {
      s->blocks.push_back(hit[j]);
      for (int64_t i = 0; i < bs; ++i) *slot++ = -1;  // already stored
      cached += static_cast<int>(bs);
    } else {
      const int32_t b = a->take_block();
      s->blocks.push_back(b);
      for (int64_t i = 0; i < bs; ++i) *slot++ = static_cast<int64_t>(b) * bs + i;
      if (s->tracked) a->register_block(b, keys[j], t);
    }
    pos += bs;
  }
  if (tail > 0) {
    const int32_t b = a->take_block();
    s->blocks.push_back(b);
    for (int64_t i = 0; i < tail; ++i, ++pos) *slot++ = static_cast<int64_t>(b) * bs + pos % bs;
  }
  // the sequence's prefix state
  if (s->tracked) {
    if (nfull > 0) s->last_key = keys[nfull - 1];
    else if (head_closes) s->last_key = head_key;
    if (head_closes || nfull > 0) s->tail.clear();
    if (!head_closes && nfull == 0 && tail == 0) {
      s->tail.insert(s->tail.end(), token_ids, token_ids + head);  // the open block grew, still partial
    } else if (tail > 0) {
      s->tail.assign(token_ids + n_tokens - tail, token_ids + n_tokens);
    }
  }
  s->len = len1;
  *cached_out = cached;
  return PKV_OK;
}

int pkv_prefix_cache_stats(const pkv_alloc *a, int64_t *registered_blocks, int64_t *evictable_blocks) {
  if (!a || !registered_blocks || !evictable_blocks) return PKV_ERR_ARG;
  *registered_blocks = static_cast<int64_t>(a->cache.size());
  *evictable_blocks = static_cast<int64_t>(a->evictable.size());
  return PKV_OK;
}

int pkv_seq_append_batch(pkv_alloc *a, const int64_t *seq_ids, int n, int n_tokens, int64_t *slots_out) {
  if (!a || n < 0 || n_tokens < 0) return PKV_ERR_ARG;
  if (n == 0 || n_tokens == 0) return PKV_OK;
  if (!seq_ids || !slots_out) return PKV_ERR_ARG;
  // validate all, and count the blocks all of them need, before changing anything
  const int64_t bs = a->block_size;
  int64_t need = 0;
  if (n > 32) {  // each sequence once: sorted copy for large batches, pairwise below
    std::vector<int64_t> ids(seq_ids, seq_ids + n);
    std::sort(ids.begin(), ids.end());
    if (std::adjacent_find(ids.begin(), ids.end()) != ids.end()) return PKV_ERR_ARG;
  }
  for (int i = 0; i < n; ++i) {
    const Sequence *s = a->find(seq_ids[i]);
    if (!s || s->swapped) return PKV_ERR_ARG;
    for (int j = 0; n <= 32 && j < i; ++j)
      if (seq_ids[j] == seq_ids[i]) return PKV_ERR_ARG;
    if (s->len % bs != 0 && a->refcount[s->blocks.back()] > 1) return PKV_ERR_SHARED;
    need += a->blocks_for(s->len + n_tokens) - static_cast<int64_t>(s->blocks.size());
  }
  if (need > a->available()) return PKV_ERR_OOM;
  for (int i = 0; i < n; ++i) {
    const int rc = pkv_seq_append(a, seq_ids[i], n_tokens, slots_out + static_cast<size_t>(i) * n_tokens);
    if (rc != PKV_OK) return rc;  // cannot happen after the checks above
  }
  return PKV_OK;
}

int pkv_seq_fork(pkv_alloc *a, int64_t parent, int64_t child) {
  if (!a) return PKV_ERR_ARG;
  const Sequence *p = a->find(parent);
  if (!p || p->swapped || a->find(child)) return PKV_ERR_ARG;
  Sequence c = *p;  // copy before the map may rehash
  for (int32_t b : c.blocks) a->refcount[b] += 1;
  a->seqs.emplace(child, std::move(c));
  return PKV_OK;
}

int pkv_seq_cow(pkv_alloc *a, int64_t seq_id, int logical_block, int32_t *pair_out, int *copied) {
  if (!a || !pair_out || !copied) return PKV_ERR_ARG;
  Sequence *s = a->find(seq_id);
  if (!s || s->swapped) return PKV_ERR_ARG;
  *copied = 0;
  int64_t logical = logical_block;
  if (logical == -1) {
    if (s->len % a->block_size == 0) return PKV_OK;
    logical = s->len / a->block_size;
  }
  if (logical < 0 || logical >= static_cast<int64_t>(s->blocks.size())) return PKV_ERR_RANGE;
  const int32_t old_b = s->blocks[logical];
  if (a->refcount[old_b] <= 1) return PKV_OK;
  if (a->available() == 0) return PKV_ERR_OOM;
  const int32_t new_b = a->take_block();
  a->refcount[old_b] -= 1;  // still held by another sequence: never reaches 0 here
  s->blocks[logical] = new_b;
  pair_out[0] = old_b;
  pair_out[1] = new_b;
  *copied = 1;
  return PKV_OK;
}

int pkv_seq_free(pkv_alloc *a, int64_t seq_id) {
  if (!a) return PKV_ERR_ARG;
  auto it = a->seqs.find(seq_id);
  if (it == a->seqs.end()) return PKV_ERR_ARG;
  for (int32_t b : it->second.blocks) a->release_block(b);
  a->seqs.erase(it);
  return PKV_OK;
}

int pkv_seq_swap_out(pkv_alloc *a, int64_t seq_id, int32_t *blocks_out, int max_blocks, int *n_out) {
  if (!a || !n_out || max_blocks < 0) return PKV_ERR_ARG;
  Sequence *s = a->find(seq_id);
  if (!s || s->swapped) return PKV_ERR_ARG;
  const int64_t nb = static_cast<int64_t>(s->blocks.size());
  if (nb > max_blocks) return PKV_ERR_RANGE;
  if (nb > 0 && !blocks_out) return PKV_ERR_ARG;
  for (int64_t i = 0; i < nb; ++i) blocks_out[i] = s->blocks[i];
  for (int32_t b : s->blocks) a->release_block(b);
  s->blocks.clear();
  s->swapped = true;
  *n_out = static_cast<int>(nb);
  return PKV_OK;
}

int pkv_seq_swap_in(pkv_alloc *a, int64_t seq_id, int32_t *blocks_out, int max_blocks, int *n_out) {
  if (!a || !n_out || max_blocks < 0) return PKV_ERR_ARG;
  Sequence *s = a->find(seq_id);
  if (!s || !s->swapped) return PKV_ERR_ARG;
  const int64_t nb = a->blocks_for(s->len);
  if (nb > max_blocks) return PKV_ERR_RANGE;
  if (nb > 0 && !blocks_out) return PKV_ERR_ARG;
  if (nb > a->available()) return PKV_ERR_OOM;
  for (int64_t i = 0; i < nb; ++i) {
    const int32_t b = a->take_block();
    s->blocks.push_back(b);
    blocks_out[i] = b;
  }
  s->swapped = false;
  s->tracked = false;  // fresh blocks, not registered
  s->tail.clear();
  *n_out = static_cast<int>(nb);
  return PKV_OK;
}

int64_t pkv_seq_len(const pkv_alloc *a, int64_t seq_id) {
  if (!a) return PKV_ERR_ARG;
  const Sequence *s = a->find(seq_id);
  return s ? s->len : PKV_ERR_ARG;
}

int pkv_block_table(const pkv_alloc *a, const int64_t *seq_ids, int n, int32_t *table_out,
                    int max_blocks, int32_t *lens_out) {
  if (!a || n < 0 || max_blocks < 0 || (n > 0 && (!seq_ids || !table_out || !lens_out)))
    return PKV_ERR_ARG;
  for (int i = 0; i < n; ++i) {  // validate everything before writing
    const Sequence *s = a->find(seq_ids[i]);
    if (!s || s->swapped) return PKV_ERR_ARG;
    if (static_cast<int64_t>(s->blocks.size()) > max_blocks) return PKV_ERR_RANGE;
    if (s->len > INT32_MAX) return PKV_ERR_RANGE;
  }
  for (int i = 0; i < n; ++i) {
    const Sequence *s = a->find(seq_ids[i]);
    int32_t *row = table_out + static_cast<size_t>(i) * max_blocks;
    const size_t nb = s->blocks.size();
    if (nb) std::memcpy(row, s->blocks.data(), nb * sizeof(int32_t));
    for (size_t j = nb; j < static_cast<size_t>(max_blocks); ++j) row[j] = -1;
    lens_out[i] = static_cast<int32_t>(s->len);
  }
  return PKV_OK;
}

int pkv_num_free(const pkv_alloc *a) {
  return a ? static_cast<int>(a->available()) : PKV_ERR_ARG;
}

int pkv_refcount(const pkv_alloc *a, int block) {
  if (!a) return PKV_ERR_ARG;
  if (block < 0 || block >= a->num_blocks) return PKV_ERR_RANGE;
  return a->refcount[block];
}

}  // extern "C"
