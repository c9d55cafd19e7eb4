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
// Every mutating call validates first and mutates last, so a failing call
// leaves the state unchanged.
#include <cstdint>
#include <cstring>
#include <new>
#include <unordered_map>
#include <vector>

#include "pkv.h"

namespace {

struct Sequence {
  std::vector<int32_t> blocks;  // logical -> physical
  int64_t len = 0;              // tokens stored
  bool swapped = false;         // blocks released to the pool, contents held by the caller
};

}  // namespace

struct pkv_alloc {
  int32_t num_blocks = 0;
  int32_t block_size = 0;
  std::vector<int32_t> free_stack;  // top = back()
  std::vector<int32_t> refcount;
  std::unordered_map<int64_t, Sequence> seqs;

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
  if (need > static_cast<int64_t>(a->free_stack.size())) return PKV_ERR_OOM;
  for (int64_t i = 0; i < need; ++i) {
    const int32_t b = a->free_stack.back();
    a->free_stack.pop_back();
    a->refcount[b] = 1;
    s->blocks.push_back(b);
  }
  for (int64_t pos = s->len, i = 0; pos < new_len; ++pos, ++i)
    slots_out[i] = static_cast<int64_t>(s->blocks[pos / bs]) * bs + pos % bs;
  s->len = new_len;
  return PKV_OK;
}

int pkv_seq_append_batch(pkv_alloc *a, const int64_t *seq_ids, int n, int n_tokens, int64_t *slots_out) {
  if (!a || n < 0 || n_tokens < 0) return PKV_ERR_ARG;
  if (n == 0 || n_tokens == 0) return PKV_OK;
  if (!seq_ids || !slots_out) return PKV_ERR_ARG;
  // validate all, and count the blocks all of them need, before changing anything
  const int64_t bs = a->block_size;
  int64_t need = 0;
  for (int i = 0; i < n; ++i) {
    const Sequence *s = a->find(seq_ids[i]);
    if (!s || s->swapped) return PKV_ERR_ARG;
    for (int j = 0; j < i; ++j)
      if (seq_ids[j] == seq_ids[i]) return PKV_ERR_ARG;  // each sequence once
    if (s->len % bs != 0 && a->refcount[s->blocks.back()] > 1) return PKV_ERR_SHARED;
    need += a->blocks_for(s->len + n_tokens) - static_cast<int64_t>(s->blocks.size());
  }
  if (need > static_cast<int64_t>(a->free_stack.size())) return PKV_ERR_OOM;
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
  if (a->free_stack.empty()) return PKV_ERR_OOM;
  const int32_t new_b = a->free_stack.back();
  a->free_stack.pop_back();
  a->refcount[new_b] = 1;
  a->refcount[old_b] -= 1;
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
  for (int32_t b : it->second.blocks) {
    if (--a->refcount[b] == 0) a->free_stack.push_back(b);
  }
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
  for (int32_t b : s->blocks) {
    if (--a->refcount[b] == 0) a->free_stack.push_back(b);
  }
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
  if (nb > static_cast<int64_t>(a->free_stack.size())) return PKV_ERR_OOM;
  for (int64_t i = 0; i < nb; ++i) {
    const int32_t b = a->free_stack.back();
    a->free_stack.pop_back();
    a->refcount[b] = 1;
    s->blocks.push_back(b);
    blocks_out[i] = b;
  }
  s->swapped = false;
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
  return a ? static_cast<int>(a->free_stack.size()) : PKV_ERR_ARG;
}

int pkv_refcount(const pkv_alloc *a, int block) {
  if (!a) return PKV_ERR_ARG;
  if (block < 0 || block >= a->num_blocks) return PKV_ERR_RANGE;
  return a->refcount[block];
}

}  // extern "C"
