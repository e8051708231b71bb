// block_manager.cpp -- host-side manager of the paged KV cache's blocks: the
// step that produces the attention calls' block tables and slot mappings.
//
// What it implements (the pages' statement of it):
//  - a pool of fixed 256-token blocks handed out from the front of a deque
//    of free blocks, ceil(tokens / 256) per sequence (intelliparadigm.com
//    Nano-vLLM article §2.1 动态分块内存管理, DynamicMemoryPool);
//  - direct reference counting instead of a reclaim pass (blog.hotdry.top
//    "1200行代码挑战vLLM" §2 内存管理策略: 简化回收 ... 直接引用计数);
//  - a prefix cache keyed by a hash of the prompt: a request whose prompt
//    starts with an already cached prefix reuses its K/V instead of
//    recomputing it (same article, §性能优化 1 前缀缓存);
//  - blocks of that prefix shared by every sequence that has it, each
//    sequence reaching them through its block table (ocdem.com nano-vllm
//    article §2.1 "基石PagedAttention": 块表, 高效的内存共享);
//  - delayed release (intelliparadigm.com article §7.2 延迟释放策略): a block
//    whose count drops to zero goes to the back of the free deque but keeps
//    its cached content until it is handed out again, so a later request with
//    the same prefix still finds it.
// Readings where the pages are silent: the prefix cache works at block
// granularity (a full block is cached under the hash of its 256 token ids
// chained with the key of the block before it, so a key names the whole
// prefix up to the block's end); a hit is confirmed by comparing the block's
// stored token ids and its predecessor's key, so two different prefixes can
// share a block only if their 64-bit chained keys collide; a partial block is
// never cached; only the leading run of cached blocks is reused (the K/V of a
// block depends on every token before it); a sequence's blocks are released
// from its last to its first, so the leading blocks of a prefix, the ones most
// often shared, are the last to be handed out again; an allocation that does
// not fit fails and changes nothing (the pages' fallback, a fresh device
// allocation, has no place in a fixed pool).
//
// Not thread-safe: the caller serialises calls on one manager.
#include <climits>
#include <cstdint>
#include <cstring>
#include <iterator>
#include <list>
#include <new>
#include <unordered_map>
#include <vector>

#include "pkv.h"

namespace {

constexpr int kTokensPerBlock = 256;

// Key of a full block: FNV-1a's xor-then-multiply step (64-bit offset basis
// and prime) taken over 32-bit words instead of bytes -- the predecessor's
// key (two words) then the block's 256 token ids.  It only indexes the cache:
// a hit is confirmed by comparing the stored ids and predecessor key.
uint64_t block_key(uint64_t prev, const int32_t* tokens) {
  constexpr uint64_t kPrime = 0x100000001b3ull;
  uint64_t h = 0xcbf29ce484222325ull;
  h = (h ^ (prev & 0xffffffffull)) * kPrime;
  h = (h ^ (prev >> 32)) * kPrime;
  for (int i = 0; i < kTokensPerBlock; ++i)
    h = (h ^ static_cast<uint32_t>(tokens[i])) * kPrime;
  return h;
}

struct Block {
  int32_t ref = 0;
  bool cached = false;       // holds a full block registered in the prefix cache
  uint64_t key = 0;          // its key (valid when cached)
  uint64_t prev_key = 0;     // key of the block before it in its prefix (0: first block)
  std::vector<int32_t> ids;  // its token ids (when cached)
  bool free = true;
  std::list<int32_t>::iterator pos;  // position in the free list (when free)
};

struct Sequence {
  std::vector<int32_t> table;  // physical blocks, logical order
  int32_t num_tokens = 0;
  std::vector<int32_t> tail;   // token ids of the last, partial block
  uint64_t last_full_key = 0;  // key of the last full block (0: none)
  uint64_t stamp = 0;          // last batch call that named it (duplicate check)
};

}  // namespace

struct pkv_block_manager {
  std::vector<Block> blocks;
  std::list<int32_t> free_list;  // front: next to hand out; back: last released
  std::unordered_map<uint64_t, int32_t> cache;  // key -> block
  std::unordered_map<int64_t, Sequence> seqs;
  uint64_t calls = 0;                    // batch calls so far (stamps)
  mutable std::vector<Sequence*> batch;  // scratch of the batch calls, reused

  // Hands out the free block at the front; it loses any cached content.
  int32_t take_front() {
    const int32_t b = free_list.front();
    free_list.pop_front();
    Block& blk = blocks[b];
    blk.free = false;
    if (blk.cached) {
      auto it = cache.find(blk.key);
      if (it != cache.end() && it->second == b) cache.erase(it);
      blk.cached = false;
      blk.ids.clear();
    }
    blk.ref = 1;
    return b;
  }

  // Takes a cached block for one more sequence (out of the free list if it
  // was released).
  void share(int32_t b) {
    Block& blk = blocks[b];
    if (blk.free) {
      free_list.erase(blk.pos);
      blk.free = false;
    }
    ++blk.ref;
  }

  void release(int32_t b) {
    Block& blk = blocks[b];
    if (--blk.ref == 0) {
      free_list.push_back(b);
      blk.pos = std::prev(free_list.end());
      blk.free = true;
    }
  }

  // Registers a full block under its key, unless the key already names
  // another block (which then stays the cached one).  Never throws: if the
  // host heap is exhausted the block is simply left uncached.
  void register_full(int32_t b, uint64_t prev, const int32_t* ids, uint64_t key) noexcept {
    Block& blk = blocks[b];
    try {
      if (cache.count(key)) return;
      blk.ids.assign(ids, ids + kTokensPerBlock);
      cache.emplace(key, b);
    } catch (...) {
      blk.ids.clear();
      return;
    }
    blk.cached = true;
    blk.key = key;
    blk.prev_key = prev;
  }

  // Appends one token to a sequence that has room for it (a free block if its
  // last block is full); returns the token's slot.
  int32_t append_one(Sequence& seq, int32_t token) {
    if (seq.num_tokens % kTokensPerBlock == 0)  // the last block is full: open a new one
      seq.table.push_back(take_front());
    const int32_t b = seq.table.back();
    const int32_t slot = b * kTokensPerBlock + seq.num_tokens % kTokensPerBlock;
    seq.tail.push_back(token);
    ++seq.num_tokens;
    if (seq.num_tokens % kTokensPerBlock == 0) {  // the block just became full: cache it
      const uint64_t key = block_key(seq.last_full_key, seq.tail.data());
      register_full(b, seq.last_full_key, seq.tail.data(), key);
      seq.last_full_key = key;
      seq.tail.clear();
    }
    return slot;
  }

  // The cached block holding exactly these ids after the prefix `prev`, or -1.
  int32_t lookup(uint64_t prev, const int32_t* ids, uint64_t key) const {
    auto it = cache.find(key);
    if (it == cache.end()) return -1;
    const Block& blk = blocks[it->second];
    if (blk.prev_key != prev ||
        std::memcmp(blk.ids.data(), ids, sizeof(int32_t) * kTokensPerBlock) != 0)
      return -1;
    return it->second;
  }
};

extern "C" {

pkv_status pkv_bm_create(int32_t num_blocks, pkv_block_manager** out) {
  if (!out || num_blocks <= 0 || num_blocks > INT32_MAX / kTokensPerBlock)
    return PKV_ERR_INVALID_ARG;
  *out = nullptr;
  pkv_block_manager* bm = new (std::nothrow) pkv_block_manager;
  if (!bm) return PKV_ERR_NO_MEMORY;
  try {
    bm->blocks.resize(num_blocks);
    for (int32_t b = 0; b < num_blocks; ++b) {
      bm->free_list.push_back(b);
      bm->blocks[b].pos = std::prev(bm->free_list.end());
    }
  } catch (...) {
    delete bm;
    return PKV_ERR_NO_MEMORY;
  }
  *out = bm;
  return PKV_OK;
}

void pkv_bm_destroy(pkv_block_manager* bm) { delete bm; }

int32_t pkv_bm_num_free_blocks(const pkv_block_manager* bm) {
  return bm ? static_cast<int32_t>(bm->free_list.size()) : 0;
}

pkv_status pkv_bm_allocate(pkv_block_manager* bm, int64_t seq_id, const int32_t* tokens,
                           int32_t num_tokens, int32_t* num_cached_tokens) {
  if (!bm || num_tokens < 0 || (num_tokens > 0 && !tokens)) return PKV_ERR_INVALID_ARG;
  if (bm->seqs.count(seq_id)) return PKV_ERR_INVALID_ARG;
  const int32_t nblk = (num_tokens + kTokensPerBlock - 1) / kTokensPerBlock;
  const int32_t nfull = num_tokens / kTokensPerBlock;
  try {
    // Plan first (nothing changes if the allocation does not fit): the
    // leading full blocks found in the prefix cache, then fresh blocks.
    std::vector<uint64_t> keys(nfull);
    std::vector<int32_t> hits;
    uint64_t prev = 0;
    bool hitting = true;
    int32_t fresh_from_free = 0;  // cached blocks taken out of the free list
    for (int32_t i = 0; i < nfull; ++i) {
      const int32_t* ids = tokens + static_cast<int64_t>(i) * kTokensPerBlock;
      keys[i] = block_key(prev, ids);
      if (hitting) {
        const int32_t b = bm->lookup(prev, ids, keys[i]);
        if (b >= 0) {
          hits.push_back(b);
          fresh_from_free += bm->blocks[b].free ? 1 : 0;
        } else {
          hitting = false;
        }
      }
      prev = keys[i];
    }
    const int32_t need = nblk - static_cast<int32_t>(hits.size());
    if (need + fresh_from_free > static_cast<int32_t>(bm->free_list.size()))
      return PKV_ERR_NO_MEMORY;
    // Every allocation happens before the pool changes, so a failure of the
    // host heap leaves the manager as it was.
    Sequence fresh;
    fresh.table.reserve(nblk);
    fresh.tail.reserve(kTokensPerBlock);
    fresh.tail.assign(tokens + static_cast<int64_t>(nfull) * kTokensPerBlock, tokens + num_tokens);
    Sequence& seq = bm->seqs.emplace(seq_id, std::move(fresh)).first->second;
    for (int32_t b : hits) {
      bm->share(b);
      seq.table.push_back(b);
    }
    prev = hits.empty() ? 0 : keys[hits.size() - 1];
    for (int32_t i = static_cast<int32_t>(hits.size()); i < nblk; ++i) {
      const int32_t b = bm->take_front();
      seq.table.push_back(b);
      if (i < nfull) {
        bm->register_full(b, prev, tokens + static_cast<int64_t>(i) * kTokensPerBlock, keys[i]);
        prev = keys[i];
      }
    }
    seq.num_tokens = num_tokens;
    seq.last_full_key = nfull > 0 ? keys[nfull - 1] : 0;
    if (num_cached_tokens)
      *num_cached_tokens = static_cast<int32_t>(hits.size()) * kTokensPerBlock;
  } catch (...) {
    return PKV_ERR_NO_MEMORY;
  }
  return PKV_OK;
}

pkv_status pkv_bm_append(pkv_block_manager* bm, int64_t seq_id, const int32_t* tokens,
                         int32_t n, int32_t* slots) {
  if (!bm || n < 0 || (n > 0 && !tokens)) return PKV_ERR_INVALID_ARG;
  auto it = bm->seqs.find(seq_id);
  if (it == bm->seqs.end()) return PKV_ERR_INVALID_ARG;
  Sequence& seq = it->second;
  const int64_t total = static_cast<int64_t>(seq.num_tokens) + n;
  if (total > INT32_MAX) return PKV_ERR_INVALID_ARG;
  const int64_t need = (total + kTokensPerBlock - 1) / kTokensPerBlock -
                       static_cast<int64_t>(seq.table.size());
  if (need > static_cast<int64_t>(bm->free_list.size())) return PKV_ERR_NO_MEMORY;
  try {
    seq.table.reserve(seq.table.size() + need);
    seq.tail.reserve(kTokensPerBlock);
    for (int32_t i = 0; i < n; ++i) {
      const int32_t slot = bm->append_one(seq, tokens[i]);
      if (slots) slots[i] = slot;
    }
  } catch (...) {
    return PKV_ERR_NO_MEMORY;
  }
  return PKV_OK;
}

pkv_status pkv_bm_append_decode(pkv_block_manager* bm, const int64_t* seq_ids, int32_t num_seqs,
                                const int32_t* tokens, int32_t* slot_mapping) {
  if (!bm || num_seqs < 0) return PKV_ERR_INVALID_ARG;
  if (num_seqs == 0) return PKV_OK;
  if (!seq_ids || !tokens || !slot_mapping) return PKV_ERR_INVALID_ARG;
  try {
    // Check everything first: known, distinct ids with room for one more
    // token, and enough free blocks for the sequences whose last block is full.
    bm->batch.resize(num_seqs);
    const uint64_t stamp = ++bm->calls;
    int64_t need = 0;
    for (int32_t s = 0; s < num_seqs; ++s) {
      auto it = bm->seqs.find(seq_ids[s]);
      if (it == bm->seqs.end() || it->second.stamp == stamp ||
          it->second.num_tokens == INT32_MAX)
        return PKV_ERR_INVALID_ARG;
      it->second.stamp = stamp;
      bm->batch[s] = &it->second;
      need += it->second.num_tokens % kTokensPerBlock == 0 ? 1 : 0;
    }
    if (need > static_cast<int64_t>(bm->free_list.size())) return PKV_ERR_NO_MEMORY;
    for (int32_t s = 0; s < num_seqs; ++s) {
      Sequence& seq = *bm->batch[s];
      if (seq.num_tokens % kTokensPerBlock == 0) seq.table.reserve(seq.table.size() + 1);
      seq.tail.reserve(kTokensPerBlock);
    }
    for (int32_t s = 0; s < num_seqs; ++s)
      slot_mapping[s] = bm->append_one(*bm->batch[s], tokens[s]);
  } catch (...) {
    return PKV_ERR_NO_MEMORY;
  }
  return PKV_OK;
}

pkv_status pkv_bm_decode_step(pkv_block_manager* bm, const int64_t* seq_ids, int32_t num_seqs,
                              const int32_t* tokens, int32_t max_blocks, int32_t* slot_mapping,
                              int32_t* block_tables, int32_t* context_lens) {
  if (!bm || num_seqs < 0 || max_blocks < 0) return PKV_ERR_INVALID_ARG;
  if (num_seqs == 0) return PKV_OK;
  if (!seq_ids || !tokens || !slot_mapping || !context_lens || (max_blocks > 0 && !block_tables))
    return PKV_ERR_INVALID_ARG;
  try {
    // Everything is checked before anything changes: known, distinct ids,
    // tables that still fit max_blocks after the token, enough free blocks.
    bm->batch.resize(num_seqs);
    const uint64_t stamp = ++bm->calls;
    int64_t need = 0;
    for (int32_t s = 0; s < num_seqs; ++s) {
      auto it = bm->seqs.find(seq_ids[s]);
      if (it == bm->seqs.end() || it->second.stamp == stamp ||
          it->second.num_tokens == INT32_MAX)
        return PKV_ERR_INVALID_ARG;
      Sequence& seq = it->second;
      seq.stamp = stamp;
      bm->batch[s] = &seq;
      const bool opens = seq.num_tokens % kTokensPerBlock == 0;
      if (static_cast<int64_t>(seq.table.size()) + (opens ? 1 : 0) > max_blocks)
        return PKV_ERR_INVALID_ARG;
      need += opens ? 1 : 0;
    }
    if (need > static_cast<int64_t>(bm->free_list.size())) return PKV_ERR_NO_MEMORY;
    for (int32_t s = 0; s < num_seqs; ++s) {
      Sequence& seq = *bm->batch[s];
      if (seq.num_tokens % kTokensPerBlock == 0) seq.table.reserve(seq.table.size() + 1);
      seq.tail.reserve(kTokensPerBlock);
    }
    for (int32_t s = 0; s < num_seqs; ++s) {
      Sequence& seq = *bm->batch[s];
      slot_mapping[s] = bm->append_one(seq, tokens[s]);
      const int32_t used = static_cast<int32_t>(seq.table.size());
      int32_t* row = block_tables + static_cast<int64_t>(s) * max_blocks;
      std::memcpy(row, seq.table.data(), sizeof(int32_t) * used);
      for (int32_t i = used; i < max_blocks; ++i) row[i] = -1;
      context_lens[s] = seq.num_tokens;
    }
  } catch (...) {
    return PKV_ERR_NO_MEMORY;
  }
  return PKV_OK;
}

pkv_status pkv_bm_free(pkv_block_manager* bm, int64_t seq_id) {
  if (!bm) return PKV_ERR_INVALID_ARG;
  auto it = bm->seqs.find(seq_id);
  if (it == bm->seqs.end()) return PKV_ERR_INVALID_ARG;
  const std::vector<int32_t>& table = it->second.table;
  for (auto b = table.rbegin(); b != table.rend(); ++b) bm->release(*b);
  bm->seqs.erase(it);
  return PKV_OK;
}

pkv_status pkv_bm_block_tables(const pkv_block_manager* bm, const int64_t* seq_ids,
                               int32_t num_seqs, int32_t max_blocks, int32_t* block_tables,
                               int32_t* context_lens) {
  if (!bm || num_seqs < 0 || max_blocks < 0) return PKV_ERR_INVALID_ARG;
  if (num_seqs == 0) return PKV_OK;
  if (!seq_ids || !context_lens || (max_blocks > 0 && !block_tables)) return PKV_ERR_INVALID_ARG;
  try {
    bm->batch.resize(num_seqs);
  } catch (...) {
    return PKV_ERR_NO_MEMORY;
  }
  for (int32_t s = 0; s < num_seqs; ++s) {  // check everything before writing anything
    auto it = bm->seqs.find(seq_ids[s]);
    if (it == bm->seqs.end() || static_cast<int64_t>(it->second.table.size()) > max_blocks)
      return PKV_ERR_INVALID_ARG;
    bm->batch[s] = const_cast<Sequence*>(&it->second);
  }
  for (int32_t s = 0; s < num_seqs; ++s) {
    const Sequence& seq = *bm->batch[s];
    const int32_t used = static_cast<int32_t>(seq.table.size());
    int32_t* row = block_tables + static_cast<int64_t>(s) * max_blocks;
    if (used > 0) std::memcpy(row, seq.table.data(), sizeof(int32_t) * used);
    for (int32_t i = used; i < max_blocks; ++i) row[i] = -1;
    context_lens[s] = seq.num_tokens;
  }
  return PKV_OK;
}

pkv_status pkv_bm_slots(const pkv_block_manager* bm, int64_t seq_id, int32_t begin, int32_t end,
                        int32_t* slots) {
  if (!bm || begin < 0 || end < begin || (end > begin && !slots)) return PKV_ERR_INVALID_ARG;
  auto it = bm->seqs.find(seq_id);
  if (it == bm->seqs.end()) return PKV_ERR_INVALID_ARG;
  const Sequence& seq = it->second;
  if (end > seq.num_tokens) return PKV_ERR_INVALID_ARG;
  for (int32_t t = begin; t < end; ++t)
    slots[t - begin] = seq.table[t / kTokensPerBlock] * kTokensPerBlock + t % kTokensPerBlock;
  return PKV_OK;
}

int32_t pkv_bm_ref_count(const pkv_block_manager* bm, int32_t block) {
  if (!bm || block < 0 || block >= static_cast<int32_t>(bm->blocks.size())) return -1;
  return bm->blocks[block].ref;
}

}  // extern "C"
