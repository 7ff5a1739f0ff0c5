// Host block manager of a paged KV pool: which physical blocks hold which
// sequence's tokens.
//
// Blocks of block_size token slots are handed out from a free list. A
// sequence's block table lists its blocks in token order (token t in slot
// t % block_size of block table[t / block_size]), as in the KV cache page
// manager of the TFFInfer article (section 3.6.4) and the paged layout of the
// heterogeneous engine article (section 2.3). Blocks are reference counted so
// that sequences can share them:
//  - prefix cache: a full block is identified by the hash of its parent chain
//    and its own token ids; a sequence admitted with a prompt whose leading
//    full blocks are already cached reuses those blocks (their KV is already
//    written) instead of new ones;
//  - fork: a child sequence shares all of its parent's blocks;
//  - copy-on-write: a sequence about to write into a partly filled block that
//    another sequence also holds first gets a private copy of it (the caller
//    copies the page records: pa_copy_blocks).
// Cached blocks that no sequence holds stay cached until their slot is
// needed (least recently released first).
//
// CPU swap tier (the heterogeneous engine article, section 4.3: the block
// manager's swap_out moves GPU blocks to a CPU second-level cache and
// swap_in brings them back): a swapped-out
// sequence holds host slots instead of GPU blocks. Swapping out copies every
// block of the sequence to a slot of its own and releases the GPU blocks
// (blocks other sequences still hold stay on the GPU; an idle cached block
// stays in the prefix cache until reused); swapping in takes fresh GPU blocks
// and frees the slots. The caller moves the page records with the returned
// copy lists (pa_swap_blocks), in call order on one stream.
#include <algorithm>
#include <cstdint>
#include <list>
#include <new>
#include <unordered_map>
#include <vector>

#include "pagedattn.h"

namespace {

struct Block {
  int32_t ref = 0;              // sequences holding the block
  bool cached = false;          // registered in the prefix cache (full, hashed)
  uint64_t hash = 0;            // chain hash when cached
  uint64_t parent = 0;          // chain hash of the blocks before it
  std::vector<int32_t> tokens;  // token ids when cached (checked on a hash hit)
  std::list<int32_t>::iterator lru;  // position among idle cached blocks
};

struct Sequence {
  std::vector<int32_t> blocks;  // GPU blocks, or host slots while swapped out
  bool swapped = false;
  int64_t len = 0;
  uint64_t tail_hash = 0;       // chain hash through the last full block (0: none)
  std::vector<int32_t> tail;    // token ids of the partly filled last block (prefix cache)
};

// Bits of the chain hash kept (all by default). A build with a narrow mask
// makes collisions frequent, which the tests use to check that a hash hit
// is only taken after its token ids match.
#ifndef PA_BM_HASH_MASK
#define PA_BM_HASH_MASK 0xFFFFFFFFFFFFFFFFull
#endif

// 64-bit mix (splitmix64 finaliser) and the chain hash of one full block.
uint64_t mix64(uint64_t x) {
  x += 0x9E3779B97F4A7C15ull;
  x = (x ^ (x >> 30)) * 0xBF58476D1CE4E5B9ull;
  x = (x ^ (x >> 27)) * 0x94D049BB133111EBull;
  return x ^ (x >> 31);
}

uint64_t block_hash(uint64_t parent, const int32_t* tokens, int32_t n) {
  uint64_t h = mix64(parent ^ 0x5DEECE66Dull);
  for (int32_t i = 0; i < n; ++i) h = mix64(h ^ (uint64_t)(uint32_t)tokens[i]);
  return (h & PA_BM_HASH_MASK) | 1ull;  // never 0 (0 means "no parent")
}

}  // namespace

struct pa_block_manager {
  int32_t block_size;
  bool prefix_cache;
  std::vector<Block> blocks;
  std::vector<int32_t> free_list;                // never used or fully released, uncached
  std::list<int32_t> idle_cached;                // cached, ref == 0, oldest first
  std::unordered_map<uint64_t, int32_t> cache;   // chain hash -> block
  std::unordered_map<int64_t, Sequence> seqs;
  std::vector<int32_t> cpu_free;                 // free host slots
  int32_t cpu_blocks = 0;

  int32_t available() const { return (int32_t)(free_list.size() + idle_cached.size()); }

  // Take a block for new content: a free one, else the least recently
  // released cached one (dropped from the cache). Caller checked available().
  int32_t take() {
    int32_t b;
    if (!free_list.empty()) {
      b = free_list.back();
      free_list.pop_back();
    } else {
      b = idle_cached.front();
      idle_cached.pop_front();
      cache.erase(blocks[b].hash);
      blocks[b].cached = false;
      blocks[b].tokens.clear();
    }
    blocks[b].ref = 1;
    return b;
  }

  void hold(int32_t b) {
    if (blocks[b].ref == 0 && blocks[b].cached) idle_cached.erase(blocks[b].lru);
    ++blocks[b].ref;
  }

  void release(int32_t b) {
    if (--blocks[b].ref > 0) return;
    if (blocks[b].cached) {
      idle_cached.push_back(b);
      blocks[b].lru = std::prev(idle_cached.end());
    } else {
      free_list.push_back(b);
    }
  }

  // Cached block holding exactly `tokens` after the chain `parent`, or -1.
  int32_t lookup(uint64_t h, uint64_t parent, const int32_t* tokens) const {
    auto it = cache.find(h);
    if (it == cache.end()) return -1;
    const Block& bl = blocks[it->second];
    return bl.parent == parent && std::equal(bl.tokens.begin(), bl.tokens.end(), tokens) ? it->second : -1;
  }

  void register_full(int32_t b, uint64_t h, uint64_t parent, const int32_t* tokens) {
    if (cache.count(h)) return;  // same content already cached in another block
    blocks[b].cached = true;
    blocks[b].hash = h;
    blocks[b].parent = parent;
    blocks[b].tokens.assign(tokens, tokens + block_size);
    cache.emplace(h, b);
  }
};

extern "C" {

pa_status pa_bm_create(int32_t num_blocks, int32_t block_size, int32_t prefix_cache, pa_block_manager** out) {
  if (!out) return PA_ERR_INVALID_ARG;
  *out = nullptr;
  if (num_blocks < 1 || block_size < 1) return PA_ERR_INVALID_ARG;
  pa_block_manager* bm = new (std::nothrow) pa_block_manager();
  if (!bm) return PA_ERR_OOM;
  bm->block_size = block_size;
  bm->prefix_cache = prefix_cache != 0;
  bm->blocks.resize((size_t)num_blocks);
  bm->free_list.reserve((size_t)num_blocks);
  for (int32_t b = num_blocks - 1; b >= 0; --b) bm->free_list.push_back(b);  // hand out 0, 1, 2, ...
  *out = bm;
  return PA_OK;
}

pa_status pa_bm_destroy(pa_block_manager* bm) {
  delete bm;
  return PA_OK;
}

pa_status pa_bm_add_sequence(pa_block_manager* bm, int64_t seq_id, const int32_t* tokens, int32_t n_tokens,
                             int32_t* n_cached_tokens) {
  if (!bm || n_tokens < 0 || (n_tokens > 0 && bm->prefix_cache && !tokens)) return PA_ERR_INVALID_ARG;
  if (bm->seqs.count(seq_id)) return PA_ERR_INVALID_ARG;
  const int32_t bs = bm->block_size;
  const int64_t nblk = ((int64_t)n_tokens + bs - 1) / bs;
  const int64_t nfull = n_tokens / bs;
  // leading full blocks found in the prefix cache
  std::vector<int32_t> hits;
  uint64_t parent = 0;
  if (bm->prefix_cache) {
    for (int64_t i = 0; i < nfull; ++i) {
      const uint64_t h = block_hash(parent, tokens + i * bs, bs);
      const int32_t b = bm->lookup(h, parent, tokens + i * bs);
      if (b < 0) break;
      hits.push_back(b);
      parent = h;
    }
  }
  // blocks needed: the rest, from free or idle cached blocks (a hit on an
  // idle cached block takes it out of that pool)
  int32_t idle_hits = 0;
  for (int32_t b : hits) idle_hits += bm->blocks[b].ref == 0;
  if (nblk - (int64_t)hits.size() > (int64_t)bm->available() - idle_hits) return PA_ERR_OOM;
  Sequence sq;
  for (int32_t b : hits) {
    bm->hold(b);
    sq.blocks.push_back(b);
  }
  for (int64_t i = (int64_t)hits.size(); i < nblk; ++i) {
    const int32_t b = bm->take();
    sq.blocks.push_back(b);
    if (bm->prefix_cache && i < nfull) {
      const uint64_t h = block_hash(parent, tokens + i * bs, bs);
      bm->register_full(b, h, parent, tokens + i * bs);
      parent = h;
    }
  }
  sq.len = n_tokens;
  sq.tail_hash = parent;
  if (bm->prefix_cache) sq.tail.assign(tokens + nfull * bs, tokens + n_tokens);
  bm->seqs.emplace(seq_id, std::move(sq));
  if (n_cached_tokens) *n_cached_tokens = (int32_t)(hits.size() * (size_t)bs);
  return PA_OK;
}

pa_status pa_bm_fork(pa_block_manager* bm, int64_t parent_id, int64_t child_id) {
  if (!bm || bm->seqs.count(child_id)) return PA_ERR_INVALID_ARG;
  auto it = bm->seqs.find(parent_id);
  if (it == bm->seqs.end() || it->second.swapped) return PA_ERR_INVALID_ARG;
  Sequence child = it->second;
  for (int32_t b : child.blocks) bm->hold(b);
  bm->seqs.emplace(child_id, std::move(child));
  return PA_OK;
}

pa_status pa_bm_append_tokens(pa_block_manager* bm, int64_t seq_id, const int32_t* tokens, int32_t n_tokens,
                              int32_t* copy_src, int32_t* copy_dst, int32_t copy_capacity, int32_t* n_copies) {
  if (!bm || n_tokens < 0 || (n_tokens > 0 && bm->prefix_cache && !tokens)) return PA_ERR_INVALID_ARG;
  auto it = bm->seqs.find(seq_id);
  if (it == bm->seqs.end() || it->second.swapped) return PA_ERR_INVALID_ARG;
  Sequence& sq = it->second;
  const int32_t bs = bm->block_size;
  if (n_copies) *n_copies = 0;
  if (n_tokens == 0) return PA_OK;
  // a shared, partly filled last block is copied before it is written
  const bool cow = sq.len % bs != 0 && bm->blocks[sq.blocks.back()].ref > 1;
  if (cow && (!copy_src || !copy_dst || copy_capacity < 1 || !n_copies)) return PA_ERR_INVALID_ARG;
  const int64_t fill = sq.len % bs == 0 ? 0 : bs - sq.len % bs;  // free slots in the last block
  const int64_t fresh = n_tokens > fill ? (n_tokens - fill + bs - 1) / bs : 0;
  if ((int64_t)cow + fresh > bm->available()) return PA_ERR_OOM;
  if (cow) {
    const int32_t old = sq.blocks.back();
    const int32_t b = bm->take();
    bm->release(old);
    sq.blocks.back() = b;
    copy_src[0] = old;
    copy_dst[0] = b;
    *n_copies = 1;
  }
  for (int64_t i = 0; i < fresh; ++i) sq.blocks.push_back(bm->take());
  // blocks filled up by these tokens join the prefix cache
  const int64_t start = sq.len;
  sq.len += n_tokens;
  if (bm->prefix_cache) {
    for (int32_t i = 0; i < n_tokens; ++i) {
      sq.tail.push_back(tokens[i]);
      if ((int32_t)sq.tail.size() == bs) {
        const uint64_t h = block_hash(sq.tail_hash, sq.tail.data(), bs);
        bm->register_full(sq.blocks[(size_t)((start + i) / bs)], h, sq.tail_hash, sq.tail.data());
        sq.tail_hash = h;
        sq.tail.clear();
      }
    }
  }
  return PA_OK;
}

pa_status pa_bm_free_sequence(pa_block_manager* bm, int64_t seq_id) {
  if (!bm) return PA_ERR_INVALID_ARG;
  auto it = bm->seqs.find(seq_id);
  if (it == bm->seqs.end()) return PA_ERR_INVALID_ARG;
  if (it->second.swapped) {
    for (int32_t c : it->second.blocks) bm->cpu_free.push_back(c);
  } else {
    // release tail first, so that a chain's leaf is evicted before its root
    for (auto b = it->second.blocks.rbegin(); b != it->second.blocks.rend(); ++b) bm->release(*b);
  }
  bm->seqs.erase(it);
  return PA_OK;
}

pa_status pa_bm_block_table(const pa_block_manager* bm, int64_t seq_id, int32_t* table, int32_t max_blocks,
                            int32_t* num_blocks, int64_t* seq_len) {
  if (!bm || max_blocks < 0 || (max_blocks > 0 && !table)) return PA_ERR_INVALID_ARG;
  auto it = bm->seqs.find(seq_id);
  if (it == bm->seqs.end() || it->second.swapped) return PA_ERR_INVALID_ARG;
  const Sequence& sq = it->second;
  if (num_blocks) *num_blocks = (int32_t)sq.blocks.size();
  if (seq_len) *seq_len = sq.len;
  if ((int64_t)sq.blocks.size() > max_blocks) return PA_ERR_INVALID_ARG;
  std::copy(sq.blocks.begin(), sq.blocks.end(), table);
  std::fill(table + sq.blocks.size(), table + max_blocks, -1);
  return PA_OK;
}

int32_t pa_bm_num_free_blocks(const pa_block_manager* bm) { return bm ? bm->available() : 0; }

pa_status pa_bm_set_cpu_blocks(pa_block_manager* bm, int32_t num_cpu_blocks) {
  if (!bm || num_cpu_blocks < 0) return PA_ERR_INVALID_ARG;
  if ((int32_t)bm->cpu_free.size() != bm->cpu_blocks) return PA_ERR_INVALID_ARG;  // slots in use
  bm->cpu_blocks = num_cpu_blocks;
  bm->cpu_free.clear();
  for (int32_t c = num_cpu_blocks - 1; c >= 0; --c) bm->cpu_free.push_back(c);  // hand out 0, 1, 2, ...
  return PA_OK;
}

int32_t pa_bm_num_free_cpu_blocks(const pa_block_manager* bm) { return bm ? (int32_t)bm->cpu_free.size() : 0; }

pa_status pa_bm_swap_out(pa_block_manager* bm, int64_t seq_id, int32_t* gpu_src, int32_t* cpu_dst,
                         int32_t capacity, int32_t* n_copies) {
  if (!bm || !n_copies) return PA_ERR_INVALID_ARG;
  *n_copies = 0;
  auto it = bm->seqs.find(seq_id);
  if (it == bm->seqs.end() || it->second.swapped) return PA_ERR_INVALID_ARG;
  Sequence& sq = it->second;
  const int32_t n = (int32_t)sq.blocks.size();
  if (n > 0 && (!gpu_src || !cpu_dst || capacity < n)) return PA_ERR_INVALID_ARG;
  if (n > (int32_t)bm->cpu_free.size()) return PA_ERR_OOM;
  std::vector<int32_t> slots((size_t)n);
  for (int32_t i = 0; i < n; ++i) {
    slots[(size_t)i] = bm->cpu_free.back();
    bm->cpu_free.pop_back();
    gpu_src[i] = sq.blocks[(size_t)i];
    cpu_dst[i] = slots[(size_t)i];
  }
  for (auto b = sq.blocks.rbegin(); b != sq.blocks.rend(); ++b) bm->release(*b);
  sq.blocks = std::move(slots);
  sq.swapped = true;
  *n_copies = n;
  return PA_OK;
}

pa_status pa_bm_swap_in(pa_block_manager* bm, int64_t seq_id, int32_t* cpu_src, int32_t* gpu_dst,
                        int32_t capacity, int32_t* n_copies) {
  if (!bm || !n_copies) return PA_ERR_INVALID_ARG;
  *n_copies = 0;
  auto it = bm->seqs.find(seq_id);
  if (it == bm->seqs.end() || !it->second.swapped) return PA_ERR_INVALID_ARG;
  Sequence& sq = it->second;
  const int32_t n = (int32_t)sq.blocks.size();
  if (n > 0 && (!cpu_src || !gpu_dst || capacity < n)) return PA_ERR_INVALID_ARG;
  if (n > bm->available()) return PA_ERR_OOM;
  for (int32_t i = 0; i < n; ++i) {
    const int32_t b = bm->take();
    cpu_src[i] = sq.blocks[(size_t)i];
    gpu_dst[i] = b;
    bm->cpu_free.push_back(sq.blocks[(size_t)i]);
    sq.blocks[(size_t)i] = b;
  }
  sq.swapped = false;
  *n_copies = n;
  return PA_OK;
}

pa_status pa_bm_swapped_slots(const pa_block_manager* bm, int64_t seq_id, int32_t* slots, int32_t capacity,
                              int32_t* n_slots) {
  if (!bm || !n_slots || capacity < 0 || (capacity > 0 && !slots)) return PA_ERR_INVALID_ARG;
  auto it = bm->seqs.find(seq_id);
  if (it == bm->seqs.end() || !it->second.swapped) return PA_ERR_INVALID_ARG;
  const std::vector<int32_t>& v = it->second.blocks;
  *n_slots = (int32_t)v.size();
  if ((int32_t)v.size() > capacity) return PA_ERR_INVALID_ARG;
  std::copy(v.begin(), v.end(), slots);
  return PA_OK;
}

int32_t pa_bm_ref_count(const pa_block_manager* bm, int32_t block) {
  if (!bm || block < 0 || block >= (int32_t)bm->blocks.size()) return -1;
  return bm->blocks[(size_t)block].ref;
}

}  // extern "C"
