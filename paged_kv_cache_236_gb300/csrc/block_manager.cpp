// Host block manager of the block-paged KV cache (C ABI in paged_kv_blocks.h).
//
// "Paged Attention 基础 - 原理与实现进度", section 3.1 C: a free-list block
// allocator and the [batch, max_blocks_per_seq] block table; section 1,
// problems 2 and 3: sequences grow by whole blocks and may share physical
// blocks (prefix caching).  "ADR 004: Paged Attention Serving Integration",
// Decision 5 and Consequences: tables keyed by sequence id, one update call
// for fresh and growing sequences, free(seq_id) at the end of a request;
// Limitations: add_prefix / try_get_prefix_blocks.
//
// State, all O(1) per block:
//   free_     the free list (a stack; the end is allocated next)
//   ref_      per block: how many table entries name it
//   idle_     cached blocks named by no table, oldest release first, with
//             per-block iterators for O(1) removal on a prefix hit
//   cache_    prefix entries: key (parent entry id, block_size token ids) ->
//             (entry id, block); per block the key it is cached under
//   seqs_     per sequence: block table and token count
// Every mutating call first checks that it can complete (ids, sizes, the
// blocks it needs), then applies, so a refused call changes nothing.
#include <algorithm>
#include <cstdio>
#include <cstring>
#include <iterator>
#include <list>
#include <new>
#include <unordered_map>
#include <vector>

#include "paged_kv_blocks.h"
#include "pkv_internal.h"

namespace {

struct KeyHash {
  size_t operator()(const std::vector<int64_t>& k) const noexcept {
    uint64_t h = 0x9E3779B97F4A7C15ull;
    for (int64_t v : k) {
      h ^= (uint64_t)v + 0x9E3779B97F4A7C15ull + (h << 6) + (h >> 2);
      h *= 0xBF58476D1CE4E5B9ull;
    }
    return (size_t)(h ^ (h >> 31));
  }
};

struct Seq {
  std::vector<int32_t> table;
  int64_t len = 0;
};

struct CacheEntry {
  int64_t id;
  int32_t block;
};

pkv_status fail(pkv_status st, const char* fmt, long long a = 0, long long b = 0) {
  char msg[256];
  snprintf(msg, sizeof(msg), fmt, a, b);
  pkv::set_last_error(msg);
  return st;
}

}  // namespace

struct pkv_block_manager {
  int32_t nb, bs, max_blocks;
  std::vector<int32_t> free_;
  std::vector<int32_t> ref_;
  std::list<int32_t> idle_;
  std::vector<std::list<int32_t>::iterator> idle_pos_;
  std::vector<char> is_idle_;
  std::unordered_map<std::vector<int64_t>, CacheEntry, KeyHash> cache_;
  std::vector<std::vector<int64_t>> block_key_;  // empty: not cached
  std::vector<int64_t> block_entry_;             // 0: not cached
  std::unordered_map<int64_t, Seq> seqs_;
  int64_t next_entry_ = 1;
  int32_t used_ = 0;
  // per-call scratch of pkv_bm_step, kept to avoid allocations
  std::vector<int64_t> ids_scratch_;
  std::vector<std::pair<int32_t, int32_t>> dropped_;  // (shared last block, copies made of it)

  pkv_block_manager(int32_t n, int32_t b, int32_t m)
      : nb(n), bs(b), max_blocks(m), ref_(n, 0), idle_pos_(n), is_idle_(n, 0), block_key_(n), block_entry_(n, 0) {
    free_.reserve(n);
    for (int32_t i = n - 1; i >= 0; --i) free_.push_back(i);
  }

  int64_t available() const { return (int64_t)free_.size() + (int64_t)idle_.size(); }
  int64_t blocks_for(int64_t tokens) const { return (tokens + bs - 1) / bs; }

  // Caller has checked available() > 0.
  int32_t take() {
    int32_t b;
    if (!free_.empty()) {
      b = free_.back();
      free_.pop_back();
    } else {
      b = idle_.front();
      idle_.pop_front();
      is_idle_[b] = 0;
      cache_.erase(block_key_[b]);
      block_key_[b].clear();
      block_entry_[b] = 0;
    }
    ref_[b] = 1;
    ++used_;
    return b;
  }

  void acquire(int32_t b) {
    if (ref_[b] == 0) {
      if (is_idle_[b]) {
        idle_.erase(idle_pos_[b]);
        is_idle_[b] = 0;
      }
      ++used_;
    }
    ++ref_[b];
  }

  void release(int32_t b) {
    if (--ref_[b] == 0) {
      --used_;
      if (block_entry_[b] != 0) {
        idle_.push_back(b);
        idle_pos_[b] = std::prev(idle_.end());
        is_idle_[b] = 1;
      } else {
        free_.push_back(b);
      }
    }
  }

  // Blocks an append of n tokens to s takes: the copy-on-write (if the last
  // block is partly filled and named `named` > 1 times) plus new blocks.
  int64_t need(const Seq& s, int64_t n, int32_t named, bool* cow) const {
    *cow = n > 0 && s.len % bs != 0 && named > 1;
    return (*cow ? 1 : 0) + blocks_for(s.len + n) - (int64_t)s.table.size();
  }

  // Applies an append whose blocks are known to be available.
  void append(Seq& s, int64_t n, int64_t* slots, int32_t* copy_pair, int32_t* ncopies) {
    if (n > 0 && s.len % bs != 0 && ref_[s.table.back()] > 1) {
      const int32_t src = s.table.back();
      const int32_t dst = take();
      --ref_[src];  // still >= 1: src stays in use
      s.table.back() = dst;
      copy_pair[0] = src;
      copy_pair[1] = dst;
      ++*ncopies;
    }
    while ((int64_t)s.table.size() < blocks_for(s.len + n)) s.table.push_back(take());
    for (int64_t p = s.len; p < s.len + n; ++p)
      slots[p - s.len] = (int64_t)s.table[p / bs] * bs + p % bs;
    s.len += n;
  }

  std::vector<int64_t> key_of(int64_t parent, const int64_t* tokens) const {
    std::vector<int64_t> k(bs + 1);
    k[0] = parent;
    memcpy(k.data() + 1, tokens, sizeof(int64_t) * bs);
    return k;
  }
};

extern "C" {

pkv_status pkv_bm_create(int32_t num_blocks, int32_t block_size, int32_t max_blocks_per_seq,
                         pkv_block_manager** out) {
  pkv::set_last_error("");
  if (!out) return fail(PKV_ERR_INVALID_ARG, "null handle pointer");
  *out = nullptr;
  if (num_blocks <= 0 || block_size <= 0 || max_blocks_per_seq <= 0)
    return fail(PKV_ERR_INVALID_ARG, "sizes must be positive");
  if ((int64_t)max_blocks_per_seq * block_size > ((int64_t)1 << 31) - 1)
    return fail(PKV_ERR_INVALID_ARG, "max_blocks_per_seq * block_size exceeds int32");
  *out = new (std::nothrow) pkv_block_manager(num_blocks, block_size, max_blocks_per_seq);
  if (!*out) return fail(PKV_ERR_INVALID_ARG, "out of host memory");
  return PKV_OK;
}

void pkv_bm_destroy(pkv_block_manager* bm) { delete bm; }

pkv_status pkv_bm_update(pkv_block_manager* bm, int64_t seq_id, int32_t num_new_tokens, int64_t* slot_mapping,
                         int32_t* copy_pair, int32_t* num_copies) {
  pkv::set_last_error("");
  if (!bm || !copy_pair || !num_copies) return fail(PKV_ERR_INVALID_ARG, "null pointer");
  if (num_new_tokens < 0) return fail(PKV_ERR_INVALID_ARG, "num_new_tokens < 0");
  if (num_new_tokens > 0 && !slot_mapping) return fail(PKV_ERR_INVALID_ARG, "null slot_mapping");
  *num_copies = 0;
  auto it = bm->seqs_.find(seq_id);
  Seq fresh;
  const Seq& s = it == bm->seqs_.end() ? fresh : it->second;
  if (bm->blocks_for(s.len + num_new_tokens) > bm->max_blocks)
    return fail(PKV_ERR_INVALID_ARG, "sequence %lld would need more than %lld blocks", (long long)seq_id,
                bm->max_blocks);
  bool cow;
  const int64_t need = bm->need(s, num_new_tokens, s.table.empty() ? 0 : bm->ref_[s.table.back()], &cow);
  if (need > bm->available())
    return fail(PKV_ERR_OUT_OF_BLOCKS, "need %lld blocks, %lld free or evictable", need, bm->available());
  Seq& t = bm->seqs_[seq_id];
  bm->append(t, num_new_tokens, slot_mapping, copy_pair, num_copies);
  return PKV_OK;
}

pkv_status pkv_bm_step(pkv_block_manager* bm, const int64_t* seq_ids, const int32_t* num_new_tokens,
                       int32_t num_seqs, int64_t* slot_mapping, int32_t* block_tables, int32_t* context_lens,
                       int32_t* query_start_loc, int32_t* copies, int32_t* num_copies) {
  pkv::set_last_error("");
  if (!bm || !num_copies || num_seqs < 0) return fail(PKV_ERR_INVALID_ARG, "null pointer or num_seqs < 0");
  *num_copies = 0;
  if (num_seqs == 0) {
    if (query_start_loc) query_start_loc[0] = 0;
    return PKV_OK;
  }
  if (!seq_ids || !num_new_tokens || !block_tables || !context_lens || !query_start_loc || !copies)
    return fail(PKV_ERR_INVALID_ARG, "null pointer");
  // checks: distinct ids, sizes, and the blocks the whole step takes, with
  // the copy-on-write of a block shared by several members counted as the
  // sequential updates would (each copy drops the shared block's count)
  std::vector<int64_t>& ids = bm->ids_scratch_;
  ids.assign(seq_ids, seq_ids + num_seqs);
  std::sort(ids.begin(), ids.end());
  const auto dup = std::adjacent_find(ids.begin(), ids.end());
  if (dup != ids.end()) return fail(PKV_ERR_INVALID_ARG, "sequence %lld twice in one step", (long long)*dup);
  std::vector<std::pair<int32_t, int32_t>>& dropped = bm->dropped_;
  dropped.clear();
  // copies already counted of shared block b (few: a linear scan)
  auto dropped_of = [&](int32_t b) -> int32_t* {
    for (auto& d : dropped)
      if (d.first == b) return &d.second;
    return nullptr;
  };
  int64_t total = 0, need = 0;
  for (int32_t i = 0; i < num_seqs; ++i) {
    const int64_t n = num_new_tokens[i];
    if (n < 0) return fail(PKV_ERR_INVALID_ARG, "num_new_tokens[%lld] < 0", i);
    total += n;
    auto it = bm->seqs_.find(seq_ids[i]);
    if (it == bm->seqs_.end()) {
      if (bm->blocks_for(n) > bm->max_blocks)
        return fail(PKV_ERR_INVALID_ARG, "sequence %lld would need more than %lld blocks", (long long)seq_ids[i],
                    bm->max_blocks);
      need += bm->blocks_for(n);
      continue;
    }
    const Seq& s = it->second;
    if (bm->blocks_for(s.len + n) > bm->max_blocks)
      return fail(PKV_ERR_INVALID_ARG, "sequence %lld would need more than %lld blocks", (long long)seq_ids[i],
                  bm->max_blocks);
    int32_t named = 0;
    int32_t* seen = nullptr;
    if (!s.table.empty()) {
      seen = dropped_of(s.table.back());
      named = bm->ref_[s.table.back()] - (seen ? *seen : 0);
    }
    bool cow;
    need += bm->need(s, n, named, &cow);
    if (cow) {
      if (seen)
        ++*seen;
      else
        dropped.emplace_back(s.table.back(), 1);
    }
  }
  if (total > ((int64_t)1 << 31) - 1) return fail(PKV_ERR_INVALID_ARG, "more than 2^31 - 1 new tokens");
  if (total > 0 && !slot_mapping) return fail(PKV_ERR_INVALID_ARG, "null slot_mapping");
  if (need > bm->available())
    return fail(PKV_ERR_OUT_OF_BLOCKS, "step needs %lld blocks, %lld free or evictable", need, bm->available());
  int64_t off = 0;
  query_start_loc[0] = 0;
  for (int32_t i = 0; i < num_seqs; ++i) {
    Seq& s = bm->seqs_[seq_ids[i]];
    bm->append(s, num_new_tokens[i], slot_mapping + off, copies + 2 * *num_copies, num_copies);
    off += num_new_tokens[i];
    query_start_loc[i + 1] = (int32_t)off;
    context_lens[i] = (int32_t)s.len;
    int32_t* row = block_tables + (int64_t)i * bm->max_blocks;
    const int32_t nbk = (int32_t)s.table.size();
    memcpy(row, s.table.data(), sizeof(int32_t) * nbk);
    for (int32_t j = nbk; j < bm->max_blocks; ++j) row[j] = -1;
  }
  return PKV_OK;
}

pkv_status pkv_bm_free(pkv_block_manager* bm, int64_t seq_id) {
  pkv::set_last_error("");
  if (!bm) return fail(PKV_ERR_INVALID_ARG, "null handle");
  auto it = bm->seqs_.find(seq_id);
  if (it == bm->seqs_.end()) return fail(PKV_ERR_INVALID_ARG, "unknown sequence %lld", (long long)seq_id);
  const std::vector<int32_t>& t = it->second.table;
  for (auto b = t.rbegin(); b != t.rend(); ++b) bm->release(*b);
  bm->seqs_.erase(it);
  return PKV_OK;
}

pkv_status pkv_bm_fork(pkv_block_manager* bm, int64_t parent_seq_id, int64_t child_seq_id) {
  pkv::set_last_error("");
  if (!bm) return fail(PKV_ERR_INVALID_ARG, "null handle");
  auto p = bm->seqs_.find(parent_seq_id);
  if (p == bm->seqs_.end()) return fail(PKV_ERR_INVALID_ARG, "unknown sequence %lld", (long long)parent_seq_id);
  if (bm->seqs_.count(child_seq_id)) return fail(PKV_ERR_INVALID_ARG, "sequence %lld exists", (long long)child_seq_id);
  Seq child = p->second;  // copied before the insert may move the map's nodes around
  for (int32_t b : child.table) bm->acquire(b);
  bm->seqs_.emplace(child_seq_id, std::move(child));
  return PKV_OK;
}

pkv_status pkv_bm_add_prefix(pkv_block_manager* bm, int64_t seq_id, const int64_t* token_ids, int32_t num_tokens) {
  pkv::set_last_error("");
  if (!bm) return fail(PKV_ERR_INVALID_ARG, "null handle");
  auto it = bm->seqs_.find(seq_id);
  if (it == bm->seqs_.end()) return fail(PKV_ERR_INVALID_ARG, "unknown sequence %lld", (long long)seq_id);
  const Seq& s = it->second;
  if (num_tokens != s.len)
    return fail(PKV_ERR_INVALID_ARG, "%lld tokens given, the sequence has %lld", num_tokens, s.len);
  if (num_tokens > 0 && !token_ids) return fail(PKV_ERR_INVALID_ARG, "null token_ids");
  int64_t parent = 0;
  for (int64_t j = 0; j < s.len / bm->bs; ++j) {
    std::vector<int64_t> key = bm->key_of(parent, token_ids + j * bm->bs);
    auto hit = bm->cache_.find(key);
    if (hit != bm->cache_.end()) {
      parent = hit->second.id;
      continue;
    }
    const int32_t b = s.table[j];
    int64_t id;
    if (bm->block_entry_[b] != 0) {  // cached under a key that no longer chains from the root
      id = bm->block_entry_[b];
      bm->cache_.erase(bm->block_key_[b]);
    } else {
      id = bm->next_entry_++;
    }
    bm->cache_.emplace(key, CacheEntry{id, b});
    bm->block_key_[b] = std::move(key);
    bm->block_entry_[b] = id;
    parent = id;
  }
  return PKV_OK;
}

pkv_status pkv_bm_try_get_prefix_blocks(pkv_block_manager* bm, int64_t seq_id, const int64_t* token_ids,
                                        int32_t num_tokens, int32_t* num_cached_tokens) {
  pkv::set_last_error("");
  if (!bm || !num_cached_tokens) return fail(PKV_ERR_INVALID_ARG, "null pointer");
  if (num_tokens < 0) return fail(PKV_ERR_INVALID_ARG, "num_tokens < 0");
  if (num_tokens > 0 && !token_ids) return fail(PKV_ERR_INVALID_ARG, "null token_ids");
  auto it = bm->seqs_.find(seq_id);
  if (it != bm->seqs_.end() && !it->second.table.empty())
    return fail(PKV_ERR_INVALID_ARG, "sequence %lld already has blocks", (long long)seq_id);
  std::vector<int32_t> hits;
  const int64_t limit = std::min<int64_t>(num_tokens > 0 ? (num_tokens - 1) / bm->bs : 0, bm->max_blocks);
  int64_t parent = 0;
  for (int64_t j = 0; j < limit; ++j) {
    auto hit = bm->cache_.find(bm->key_of(parent, token_ids + j * bm->bs));
    if (hit == bm->cache_.end()) break;
    parent = hit->second.id;
    hits.push_back(hit->second.block);
  }
  for (int32_t b : hits) bm->acquire(b);
  Seq& s = bm->seqs_[seq_id];
  s.table = std::move(hits);
  s.len = (int64_t)s.table.size() * bm->bs;
  *num_cached_tokens = (int32_t)s.len;
  return PKV_OK;
}

pkv_status pkv_bm_block_table(const pkv_block_manager* bm, int64_t seq_id, int32_t* table, int32_t* num_blocks,
                              int32_t* num_tokens) {
  pkv::set_last_error("");
  if (!bm) return fail(PKV_ERR_INVALID_ARG, "null handle");
  auto it = bm->seqs_.find(seq_id);
  if (it == bm->seqs_.end()) return fail(PKV_ERR_INVALID_ARG, "unknown sequence %lld", (long long)seq_id);
  const Seq& s = it->second;
  if (table) {
    for (int32_t j = 0; j < bm->max_blocks; ++j) table[j] = j < (int32_t)s.table.size() ? s.table[j] : -1;
  }
  if (num_blocks) *num_blocks = (int32_t)s.table.size();
  if (num_tokens) *num_tokens = (int32_t)s.len;
  return PKV_OK;
}

pkv_status pkv_bm_stats(const pkv_block_manager* bm, int32_t* free_blocks, int32_t* idle_blocks,
                        int32_t* used_blocks, int32_t* cached_entries) {
  pkv::set_last_error("");
  if (!bm) return fail(PKV_ERR_INVALID_ARG, "null handle");
  if (free_blocks) *free_blocks = (int32_t)bm->free_.size();
  if (idle_blocks) *idle_blocks = (int32_t)bm->idle_.size();
  if (used_blocks) *used_blocks = bm->used_;
  if (cached_entries) *cached_entries = (int32_t)bm->cache_.size();
  return PKV_OK;
}

}  // extern "C"
