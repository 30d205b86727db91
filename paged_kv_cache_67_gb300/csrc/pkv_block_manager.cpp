// pkv_block_manager.cpp -- the host-side block manager declared in
// include/pkv_block_manager.h: physical-block pool, per-sequence block
// tables, slot assignment for new tokens, and prefix sharing of full blocks.
//
// The pages' design (interview note "PagedAttention kernel: paged KV cache 与
// block table", sections 直接答案 and 面试官追问; the blog post on
// re-implementing paged attention, jsqmd.com news 887134): fixed-size blocks
// in one pool, a block table per sequence (logical block -> physical block),
// slot = block * bs + offset on the write side, a free-block queue, a map
// from a block's hash (its token ids chained with the hash of the prefix)
// to the block holding them, and an allocate call that reports how much of
// a prompt is already cached.  LRU eviction of cached blocks, left open in
// the blog, is implemented here.
//
// Exactness of sharing.  A registered block records its parent block and
// that parent's generation (bumped whenever a block is registered or
// evicted) and its own token ids; a lookup matches only when the parent is
// the block matched for the previous position with the same generation and
// every token id is equal.  A hash collision therefore never shares wrong
// data, and a child whose parent was evicted can no longer be matched.
#include <stdint.h>
#include <string.h>

#include <list>
#include <mutex>
#include <new>
#include <unordered_map>
#include <unordered_set>
#include <vector>

#include "pkv_block_manager.h"

namespace {

// 64-bit mixing step (the finaliser of the SplitMix64 generator, Steele,
// Lea and Flood, "Fast splittable pseudorandom number generators", 2014).
inline uint64_t mix64(uint64_t x) {
  x += 0x9e3779b97f4a7c15ull;
  x = (x ^ (x >> 30)) * 0xbf58476d1ce4e5b9ull;
  x = (x ^ (x >> 27)) * 0x94d049bb133111ebull;
  return x ^ (x >> 31);
}

// Hash of one full block: its token ids chained onto the prefix hash.
uint64_t block_hash(uint64_t prefix, const int64_t *tokens, int n) {
  uint64_t h = mix64(prefix ^ 0x6a09e667f3bcc909ull);
  for (int i = 0; i < n; ++i) h = mix64(h ^ static_cast<uint64_t>(tokens[i]));
  return h;
}

constexpr uint64_t kRootHash = 0x243f6a8885a308d3ull;  // prefix hash before the first block

struct Block {
  int ref = 0;                    // sequences whose table holds the block
  uint64_t gen = 0;               // bumped on every registration and eviction
  bool registered = false;        // listed in the hash map
  uint64_t hash = 0;
  int32_t parent = -1;            // block matched before this one (-1: first block)
  uint64_t parent_gen = 0;
  std::vector<int64_t> tokens;    // token ids of a registered block
  int free_list = 0;              // 0: not free, 1: unregistered free, 2: cached free
  std::list<int32_t>::iterator free_it;
};

struct Sequence {
  std::vector<int32_t> table;
  int64_t len = 0;
  std::vector<int64_t> tail;      // token ids of the last block while it is partly filled
  uint64_t chain_hash = kRootHash;  // hash of the prefix up to the last full block
  int32_t chain_block = -1;       // registered block standing for the last full block
  uint64_t chain_gen = 0;
};

}  // namespace

struct pkv_block_manager {
  std::mutex mu;
  int64_t num_blocks = 0;
  int bs = 0;
  bool prefix = false;
  std::vector<Block> blocks;
  std::list<int32_t> free_plain;   // free blocks holding nothing reusable: taken first
  std::list<int32_t> free_cached;  // free registered blocks, least recently freed first
  std::unordered_multimap<uint64_t, int32_t> by_hash;
  std::unordered_map<int64_t, Sequence> seqs;

  int64_t free_count() const { return (int64_t)free_plain.size() + (int64_t)free_cached.size(); }

  void to_free(int32_t id) {
    Block &b = blocks[id];
    if (b.registered) {
      b.free_list = 2;
      b.free_it = free_cached.insert(free_cached.end(), id);
    } else {
      b.free_list = 1;
      b.free_it = free_plain.insert(free_plain.end(), id);
    }
  }

  void off_free(int32_t id) {
    Block &b = blocks[id];
    if (b.free_list == 1) free_plain.erase(b.free_it);
    if (b.free_list == 2) free_cached.erase(b.free_it);
    b.free_list = 0;
  }

  void unregister(int32_t id) {
    Block &b = blocks[id];
    if (!b.registered) return;
    auto range = by_hash.equal_range(b.hash);
    for (auto it = range.first; it != range.second; ++it)
      if (it->second == id) {
        by_hash.erase(it);
        break;
      }
    b.registered = false;
    b.tokens.clear();
    ++b.gen;
  }

  // A fresh block for new contents (the caller checked that one is free).
  int32_t take_fresh() {
    int32_t id;
    if (!free_plain.empty()) {
      id = free_plain.front();
    } else {
      id = free_cached.front();  // least recently freed cached block: evicted
    }
    off_free(id);
    unregister(id);
    blocks[id].ref = 1;
    return id;
  }

  // Registered block holding `tokens` after the chain (parent, parent_gen), or -1.
  int32_t lookup(uint64_t h, int32_t parent, uint64_t parent_gen, const int64_t *tokens) const {
    auto range = by_hash.equal_range(h);
    for (auto it = range.first; it != range.second; ++it) {
      const Block &b = blocks[it->second];
      if (b.registered && b.parent == parent && (parent < 0 || b.parent_gen == parent_gen) &&
          memcmp(b.tokens.data(), tokens, sizeof(int64_t) * bs) == 0)
        return it->second;
    }
    return -1;
  }

  // Sequence s's block `id` has just been filled with `tokens`: register it
  // (unless an identical block already is) and advance the chain.
  void on_full(Sequence &s, int32_t id, const int64_t *tokens) {
    const uint64_t h = block_hash(s.chain_hash, tokens, bs);
    if (prefix) {
      int32_t canon = lookup(h, s.chain_block, s.chain_gen, tokens);
      if (canon < 0) {
        Block &b = blocks[id];
        b.registered = true;
        b.hash = h;
        b.parent = s.chain_block;
        b.parent_gen = s.chain_gen;
        b.tokens.assign(tokens, tokens + bs);
        ++b.gen;
        by_hash.emplace(h, id);
        canon = id;
      }
      s.chain_block = canon;
      s.chain_gen = blocks[canon].gen;
    }
    s.chain_hash = h;
  }
};

extern "C" {

PKV_API pkv_status pkv_bm_create(int64_t num_blocks, int block_size, int prefix_caching,
                                 pkv_block_manager **out) {
  if (!out || num_blocks <= 0 || num_blocks > 0x7fffffffLL || block_size <= 0)
    return PKV_ERR_INVALID_ARG;
  pkv_block_manager *bm = new (std::nothrow) pkv_block_manager();
  if (!bm) return PKV_ERR_INVALID_ARG;
  bm->num_blocks = num_blocks;
  bm->bs = block_size;
  bm->prefix = prefix_caching != 0;
  bm->blocks.resize((size_t)num_blocks);
  for (int64_t i = 0; i < num_blocks; ++i) bm->to_free((int32_t)i);
  *out = bm;
  return PKV_OK;
}

PKV_API void pkv_bm_destroy(pkv_block_manager *bm) { delete bm; }

PKV_API pkv_status pkv_bm_add_sequence(pkv_block_manager *bm, int64_t seq_id,
                                       const int64_t *token_ids, int64_t ntoken,
                                       int64_t *slot_mapping, int64_t *num_cached) {
  if (!bm || seq_id < 0 || !token_ids || ntoken <= 0) return PKV_ERR_INVALID_ARG;
  std::lock_guard<std::mutex> lock(bm->mu);
  if (bm->seqs.count(seq_id)) return PKV_ERR_INVALID_ARG;
  const int bs = bm->bs;
  const int64_t nblk = (ntoken + bs - 1) / bs;
  const int64_t nfull = ntoken / bs;
  if (nblk > 0x7fffffffLL) return PKV_ERR_INVALID_ARG;

  // 1. the longest run of leading full blocks already cached (no change yet)
  std::vector<int32_t> matched;
  uint64_t h = kRootHash;
  int32_t parent = -1;
  uint64_t parent_gen = 0;
  int64_t revive = 0;  // matched blocks that sit in the free list
  if (bm->prefix) {
    for (int64_t j = 0; j < nfull; ++j) {
      const int64_t *tok = token_ids + j * bs;
      const uint64_t hj = block_hash(h, tok, bs);
      const int32_t id = bm->lookup(hj, parent, parent_gen, tok);
      if (id < 0) break;
      matched.push_back(id);
      if (bm->blocks[id].ref == 0) ++revive;
      h = hj;
      parent = id;
      parent_gen = bm->blocks[id].gen;
    }
  }
  const int64_t fresh = nblk - (int64_t)matched.size();
  if (bm->free_count() - revive < fresh) return PKV_ERR_OUT_OF_BLOCKS;

  // 2. commit: revive / share the matched blocks, then take fresh ones
  Sequence s;
  s.table.reserve((size_t)nblk);
  for (int32_t id : matched) {
    Block &b = bm->blocks[id];
    if (b.ref == 0) bm->off_free(id);
    ++b.ref;
    s.table.push_back(id);
  }
  s.chain_hash = h;
  s.chain_block = parent;
  s.chain_gen = parent_gen;
  for (int64_t j = (int64_t)matched.size(); j < nblk; ++j) {
    const int32_t id = bm->take_fresh();
    s.table.push_back(id);
    if (j < nfull) bm->on_full(s, id, token_ids + j * bs);
  }
  s.len = ntoken;
  s.tail.assign(token_ids + nfull * bs, token_ids + ntoken);
  const int64_t cached = (int64_t)matched.size() * bs;
  if (slot_mapping) {
    for (int64_t t = 0; t < ntoken; ++t)
      slot_mapping[t] = t < cached ? -1 : (int64_t)s.table[(size_t)(t / bs)] * bs + t % bs;
  }
  if (num_cached) *num_cached = cached;
  bm->seqs.emplace(seq_id, std::move(s));
  return PKV_OK;
}

PKV_API pkv_status pkv_bm_append_tokens(pkv_block_manager *bm, const int64_t *seq_ids,
                                        const int64_t *token_ids, int B, int64_t *slot_mapping) {
  if (!bm || B < 0 || (B > 0 && (!seq_ids || !token_ids || !slot_mapping)))
    return PKV_ERR_INVALID_ARG;
  std::lock_guard<std::mutex> lock(bm->mu);
  const int bs = bm->bs;
  // validate everything and count the new blocks before changing anything
  std::unordered_set<int64_t> seen;
  int64_t need = 0;
  for (int i = 0; i < B; ++i) {
    if (seq_ids[i] < 0) continue;
    auto it = bm->seqs.find(seq_ids[i]);
    if (it == bm->seqs.end() || !seen.insert(seq_ids[i]).second) return PKV_ERR_INVALID_ARG;
    if (it->second.len % bs == 0) ++need;
  }
  if (need > bm->free_count()) return PKV_ERR_OUT_OF_BLOCKS;
  for (int i = 0; i < B; ++i) {
    if (seq_ids[i] < 0) {
      slot_mapping[i] = -1;
      continue;
    }
    Sequence &s = bm->seqs.find(seq_ids[i])->second;
    if (s.len % bs == 0) s.table.push_back(bm->take_fresh());
    const int32_t blk = s.table.back();
    slot_mapping[i] = (int64_t)blk * bs + s.len % bs;
    s.tail.push_back(token_ids[i]);
    ++s.len;
    if (s.len % bs == 0) {
      bm->on_full(s, blk, s.tail.data());
      s.tail.clear();
    }
  }
  return PKV_OK;
}

PKV_API pkv_status pkv_bm_free_sequence(pkv_block_manager *bm, int64_t seq_id) {
  if (!bm) return PKV_ERR_INVALID_ARG;
  std::lock_guard<std::mutex> lock(bm->mu);
  auto it = bm->seqs.find(seq_id);
  if (it == bm->seqs.end()) return PKV_ERR_INVALID_ARG;
  // release from the last block back: a prefix's blocks become the most
  // recently freed, so a sequence's tail is evicted before its prefix
  const std::vector<int32_t> &table = it->second.table;
  for (size_t j = table.size(); j-- > 0;) {
    Block &b = bm->blocks[table[j]];
    if (--b.ref == 0) bm->to_free(table[j]);
  }
  bm->seqs.erase(it);
  return PKV_OK;
}

PKV_API pkv_status pkv_bm_build_batch(pkv_block_manager *bm, const int64_t *seq_ids, int B,
                                      int max_blocks, int32_t tail, int32_t *block_tables,
                                      int32_t *context_lens) {
  if (!bm || B < 0 || max_blocks < 0 ||
      (B > 0 && (!seq_ids || !context_lens || (max_blocks > 0 && !block_tables))))
    return PKV_ERR_INVALID_ARG;
  std::lock_guard<std::mutex> lock(bm->mu);
  for (int i = 0; i < B; ++i) {
    if (seq_ids[i] < 0) continue;
    auto it = bm->seqs.find(seq_ids[i]);
    if (it == bm->seqs.end() || it->second.table.size() > (size_t)max_blocks ||
        it->second.len > 0x7fffffffLL)
      return PKV_ERR_INVALID_ARG;
  }
  for (int i = 0; i < B; ++i) {
    int32_t *row = block_tables + (size_t)i * max_blocks;
    size_t used = 0;
    context_lens[i] = 0;
    if (seq_ids[i] >= 0) {
      const Sequence &s = bm->seqs.find(seq_ids[i])->second;
      used = s.table.size();
      if (used) memcpy(row, s.table.data(), used * sizeof(int32_t));
      context_lens[i] = (int32_t)s.len;
    }
    for (size_t j = used; j < (size_t)max_blocks; ++j) row[j] = tail;
  }
  return PKV_OK;
}

PKV_API pkv_status pkv_bm_sequence_info(pkv_block_manager *bm, int64_t seq_id,
                                        int64_t *context_len, int *num_table_blocks,
                                        int32_t *table, int max_blocks) {
  if (!bm || max_blocks < 0 || (max_blocks > 0 && !table)) return PKV_ERR_INVALID_ARG;
  std::lock_guard<std::mutex> lock(bm->mu);
  auto it = bm->seqs.find(seq_id);
  if (it == bm->seqs.end()) return PKV_ERR_INVALID_ARG;
  const Sequence &s = it->second;
  if (context_len) *context_len = s.len;
  if (num_table_blocks) *num_table_blocks = (int)s.table.size();
  const size_t n = s.table.size() < (size_t)max_blocks ? s.table.size() : (size_t)max_blocks;
  if (n) memcpy(table, s.table.data(), n * sizeof(int32_t));
  return PKV_OK;
}

PKV_API void pkv_bm_stats(pkv_block_manager *bm, int64_t *free_blocks, int64_t *cached_blocks,
                          int64_t *live_sequences) {
  if (!bm) return;
  std::lock_guard<std::mutex> lock(bm->mu);
  if (free_blocks) *free_blocks = bm->free_count();
  if (cached_blocks) *cached_blocks = (int64_t)bm->by_hash.size();
  if (live_sequences) *live_sequences = (int64_t)bm->seqs.size();
}

PKV_API int pkv_bm_block_refcount(pkv_block_manager *bm, int64_t block) {
  if (!bm || block < 0 || block >= bm->num_blocks) return -1;
  std::lock_guard<std::mutex> lock(bm->mu);
  return bm->blocks[(size_t)block].ref;
}

}  // extern "C"
