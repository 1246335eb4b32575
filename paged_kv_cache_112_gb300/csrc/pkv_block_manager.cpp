// Host block manager of the paged KV cache: the allocator the decode path
// serves.  Host code only (no CUDA), part of libpkv's C ABI (pkv_bm_*).
//
// What it does, from the pages:
//  * a free list of interchangeable blocks and per-block reference counts
//    ("KV Cache & PagedAttention", section 4: alloc pops the free list, a
//    fork bumps the refcount, the last free returns the block);
//  * prefix sharing keyed by a chained hash: a full block is immutable and
//    is keyed by the hash of its tokens together with the hash of the block
//    before it (and the request's extra key: adapter identity, multimodal
//    inputs), so a hit certifies an identical token history; on admission
//    every hit is a refcount bump instead of prefill and allocation
//    ("gpu_paged_kv_cache", "Prefix sharing, reference counts, and
//    copy-on-write"; "PagedAttention internals", section 04).  A hit is
//    also checked token for token, so a hash collision cannot share a block;
//  * copy-on-write: an append that lands in a block held more than once
//    allocates a fresh block, reports the (old, new) pair for the device
//    copy, drops a reference to the old block and repoints the table;
//  * eviction: blocks nobody references but whose contents are cached stay
//    reusable until allocation needs them, least recently used first;
//    referenced blocks are never evicted ("PagedAttention internals",
//    section 04);
//  * a watermark of blocks admissions may not take, so that running
//    sequences can always append ("gpu_paged_kv_cache", "Reclaiming memory:
//    swap versus recompute"), and swap bookkeeping (release a sequence's
//    blocks to the host, take fresh ones on resume).
#include <algorithm>
#include <cstdint>
#include <cstring>
#include <list>
#include <mutex>
#include <unordered_map>
#include <unordered_set>
#include <vector>

#include "pkv.h"

namespace pkv {
namespace {

// splitmix64's output function (Vigna), used as the mixing step of the chain.
uint64_t mix64(uint64_t z) {
  z = (z ^ (z >> 30)) * 0xBF58476D1CE4E5B9ull;
  z = (z ^ (z >> 27)) * 0x94D049BB133111EBull;
  return z ^ (z >> 31);
}

constexpr uint64_t kGolden = 0x9E3779B97F4A7C15ull;

// Hash of a full block: its tokens chained onto the previous block's hash.
uint64_t block_hash(uint64_t parent, const int32_t* tokens, int n) {
  uint64_t h = mix64(parent + kGolden);
  for (int i = 0; i < n; ++i) h = mix64(h ^ (static_cast<uint64_t>(static_cast<uint32_t>(tokens[i])) + kGolden * (i + 1)));
  return h;
}

// The chain's start for a request's extra key.
uint64_t chain_root(uint64_t extra_key) { return mix64(extra_key ^ kGolden); }

struct Block {
  int ref = 0;
  bool cached = false;        // registered in the prefix cache (full, immutable)
  uint64_t hash = 0;
  uint64_t parent_hash = 0;
  std::vector<int32_t> tokens;  // of a cached block, for the exact check on a hit
  std::list<int>::iterator lru;  // position in the evictable list when ref == 0 and cached
};

struct Sequence {
  std::vector<int> table;       // physical blocks, logical order
  std::vector<int32_t> tokens;  // the whole history
  uint64_t root = 0;            // chain root (extra key)
  std::vector<uint64_t> hashes; // hash of each full block
  bool swapped = false;
};

}  // namespace
}  // namespace pkv

struct pkv_bm {
  std::mutex mu;
  int num_blocks = 0, block_size = 0, watermark = 0;
  // cumulative counters reported by pkv_bm_get_stats
  int64_t prompt_tokens = 0, prompt_tokens_cached = 0, evictions = 0, cow_copies = 0, swap_outs = 0,
          refusals = 0;
  std::vector<pkv::Block> blocks;
  std::vector<int> free_list;             // ref == 0 and not cached
  std::list<int> evictable;               // ref == 0 and cached; front = least recently used
  std::unordered_map<uint64_t, int> cache;  // block hash -> block
  std::unordered_map<int64_t, pkv::Sequence> seqs;
};

namespace pkv {
namespace {

int available(const pkv_bm* m) { return static_cast<int>(m->free_list.size() + m->evictable.size()); }

// Takes one block for new contents: from the free list, else the least
// recently used evictable cached block (dropped from the cache).  -1 if none.
int take_block(pkv_bm* m) {
  int b;
  if (!m->free_list.empty()) {
    b = m->free_list.back();
    m->free_list.pop_back();
  } else if (!m->evictable.empty()) {
    b = m->evictable.front();
    m->evictable.pop_front();
    ++m->evictions;
    Block& blk = m->blocks[b];
    m->cache.erase(blk.hash);
    blk.cached = false;
    blk.tokens.clear();
  } else {
    return -1;
  }
  m->blocks[b].ref = 1;
  return b;
}

// One more reference to block b (a cache hit or a fork).
void add_ref(pkv_bm* m, int b) {
  Block& blk = m->blocks[b];
  if (blk.ref == 0 && blk.cached) m->evictable.erase(blk.lru);
  ++blk.ref;
}

// One reference fewer; at zero a cached block becomes evictable (most
// recently used), any other block returns to the free list.
void drop_ref(pkv_bm* m, int b) {
  Block& blk = m->blocks[b];
  if (--blk.ref > 0) return;
  if (blk.cached) {
    m->evictable.push_back(b);
    blk.lru = std::prev(m->evictable.end());
  } else {
    m->free_list.push_back(b);
  }
}

// Registers full block `b` (logical index i of s) in the prefix cache under
// its chained hash, unless an identical block is already there.
void register_full(pkv_bm* m, Sequence& s, int i) {
  const int B = m->block_size;
  const uint64_t parent = i == 0 ? s.root : s.hashes[i - 1];
  const uint64_t h = block_hash(parent, s.tokens.data() + static_cast<size_t>(i) * B, B);
  if (static_cast<int>(s.hashes.size()) == i) s.hashes.push_back(h);
  const int b = s.table[i];
  Block& blk = m->blocks[b];
  if (blk.cached || m->cache.count(h)) return;
  blk.cached = true;
  blk.hash = h;
  blk.parent_hash = parent;
  blk.tokens.assign(s.tokens.begin() + static_cast<size_t>(i) * B, s.tokens.begin() + static_cast<size_t>(i + 1) * B);
  m->cache.emplace(h, b);
}

// A cached block with this history, or -1 (the tokens are compared, so a
// hash collision never shares a block).
int lookup(const pkv_bm* m, uint64_t h, uint64_t parent, const int32_t* tokens) {
  const auto it = m->cache.find(h);
  if (it == m->cache.end()) return -1;
  const Block& blk = m->blocks[it->second];
  if (blk.parent_hash != parent ||
      std::memcmp(blk.tokens.data(), tokens, sizeof(int32_t) * static_cast<size_t>(m->block_size)) != 0)
    return -1;
  return it->second;
}

// Appends `token` to s (lock held): a fresh block when the tail is full, a
// copy-on-write when it is shared.  -PKV_ERR_OUT_OF_BLOCKS (nothing changed)
// when no block can be taken.
int append_locked(pkv_bm* m, Sequence& s, int32_t token, int32_t* slot, int32_t* cow_src, int32_t* cow_dst) {
  const int B = m->block_size;
  const int pos = static_cast<int>(s.tokens.size());
  *cow_src = *cow_dst = -1;
  if (pos % B == 0) {  // the tail is full (or there is none): a fresh block
    const int b = take_block(m);
    if (b < 0) return -PKV_ERR_OUT_OF_BLOCKS;
    s.table.push_back(b);
  } else {
    const int tail = s.table[pos / B];
    if (m->blocks[tail].ref > 1) {  // shared tail: copy-on-write
      const int b = take_block(m);
      if (b < 0) return -PKV_ERR_OUT_OF_BLOCKS;
      drop_ref(m, tail);
      s.table[pos / B] = b;
      *cow_src = tail;
      *cow_dst = b;
      ++m->cow_copies;
    }
  }
  s.tokens.push_back(token);
  *slot = s.table[pos / B] * B + pos % B;
  if ((pos + 1) % B == 0) register_full(m, s, pos / B);
  return PKV_OK;
}

}  // namespace
}  // namespace pkv

using namespace pkv;

extern "C" {

int64_t pkv_pool_blocks(uint64_t kv_bytes, int num_layers, int block_size, int num_kv_heads, int head_dim,
                        int elem_bytes, int with_scales) {
  if (num_layers <= 0 || block_size <= 0 || num_kv_heads <= 0 || head_dim <= 0 || elem_bytes <= 0) return -1;
  // K and V rows of every layer for block_size tokens, plus (FP8 pools) a K
  // and a V float scale per layer and KV head.
  const uint64_t rows = 2ull * static_cast<uint64_t>(num_layers) * static_cast<uint64_t>(num_kv_heads);
  const uint64_t per_block = rows * static_cast<uint64_t>(block_size) * static_cast<uint64_t>(head_dim) *
                                 static_cast<uint64_t>(elem_bytes) +
                             (with_scales ? rows * 4ull : 0ull);
  return static_cast<int64_t>(kv_bytes / per_block);
}

pkv_bm* pkv_bm_create(int num_blocks, int block_size, int watermark_blocks) {
  if (num_blocks <= 0 || block_size <= 0 || watermark_blocks < 0 || watermark_blocks > num_blocks) return nullptr;
  // slots (block * block_size + offset) are int32
  if (static_cast<int64_t>(num_blocks) * block_size > INT32_MAX) return nullptr;
  pkv_bm* m = new pkv_bm();
  m->num_blocks = num_blocks;
  m->block_size = block_size;
  m->watermark = watermark_blocks;
  m->blocks.resize(num_blocks);
  m->free_list.reserve(num_blocks);
  for (int b = num_blocks - 1; b >= 0; --b) m->free_list.push_back(b);  // block 0 first
  return m;
}

void pkv_bm_destroy(pkv_bm* m) { delete m; }

int pkv_bm_available_blocks(pkv_bm* m) {
  if (!m) return -PKV_ERR_INVALID_ARG;
  std::lock_guard<std::mutex> lock(m->mu);
  return available(m);
}

int pkv_bm_cached_blocks(pkv_bm* m) {
  if (!m) return -PKV_ERR_INVALID_ARG;
  std::lock_guard<std::mutex> lock(m->mu);
  return static_cast<int>(m->cache.size());
}

int pkv_bm_block_refcount(pkv_bm* m, int block) {
  if (!m) return -PKV_ERR_INVALID_ARG;
  std::lock_guard<std::mutex> lock(m->mu);
  if (block < 0 || block >= m->num_blocks) return -PKV_ERR_INVALID_ARG;
  return m->blocks[block].ref;
}

int pkv_bm_add_sequence(pkv_bm* m, int64_t seq_id, const int32_t* tokens, int num_tokens, uint64_t extra_key,
                        int32_t* slots) {
  if (!m) return -PKV_ERR_INVALID_ARG;
  std::lock_guard<std::mutex> lock(m->mu);
  if (num_tokens < 0 || (num_tokens > 0 && (!tokens || !slots)) || m->seqs.count(seq_id)) return -PKV_ERR_INVALID_ARG;
  const int B = m->block_size;
  Sequence s;
  s.root = chain_root(extra_key);
  s.tokens.assign(tokens, tokens + num_tokens);
  // Cached prefix: whole blocks from position 0 whose chained hash hits.
  std::vector<int> hits;
  uint64_t parent = s.root;
  for (int i = 0; (i + 1) * B <= num_tokens; ++i) {
    const uint64_t h = block_hash(parent, tokens + static_cast<size_t>(i) * B, B);
    const int b = lookup(m, h, parent, tokens + static_cast<size_t>(i) * B);
    if (b < 0) break;
    hits.push_back(b);
    s.hashes.push_back(h);
    parent = h;
  }
  const int need = (num_tokens + B - 1) / B - static_cast<int>(hits.size());
  // Blocks a hit takes out of the evictable list are not available either.
  int hit_evictable = 0;
  for (int b : hits) hit_evictable += m->blocks[b].ref == 0 ? 1 : 0;
  if (need > available(m) - hit_evictable - m->watermark) {
    ++m->refusals;
    return -PKV_ERR_OUT_OF_BLOCKS;
  }
  for (int b : hits) {
    add_ref(m, b);
    s.table.push_back(b);
  }
  for (int i = 0; i < need; ++i) s.table.push_back(take_block(m));
  const int cached_tokens = static_cast<int>(hits.size()) * B;
  m->prompt_tokens += num_tokens;
  m->prompt_tokens_cached += cached_tokens;
  for (int t = 0; t < num_tokens; ++t)
    slots[t] = t < cached_tokens ? -1 : s.table[t / B] * B + t % B;
  // The prompt's new full blocks become cacheable once written.
  for (int i = static_cast<int>(hits.size()); (i + 1) * B <= num_tokens; ++i) register_full(m, s, i);
  m->seqs.emplace(seq_id, std::move(s));
  return cached_tokens;
}

int pkv_bm_fork(pkv_bm* m, int64_t parent, int64_t child) {
  if (!m) return -PKV_ERR_INVALID_ARG;
  std::lock_guard<std::mutex> lock(m->mu);
  const auto it = m->seqs.find(parent);
  if (it == m->seqs.end() || it->second.swapped || m->seqs.count(child)) return -PKV_ERR_INVALID_ARG;
  Sequence c = it->second;
  for (int b : c.table) add_ref(m, b);
  m->seqs.emplace(child, std::move(c));
  return PKV_OK;
}

int pkv_bm_append(pkv_bm* m, int64_t seq_id, int32_t token, int32_t* slot, int32_t* cow_src, int32_t* cow_dst) {
  if (!m) return -PKV_ERR_INVALID_ARG;
  std::lock_guard<std::mutex> lock(m->mu);
  const auto it = m->seqs.find(seq_id);
  if (it == m->seqs.end() || it->second.swapped || !slot || !cow_src || !cow_dst) return -PKV_ERR_INVALID_ARG;
  const int rc = append_locked(m, it->second, token, slot, cow_src, cow_dst);
  if (rc == -PKV_ERR_OUT_OF_BLOCKS) ++m->refusals;
  return rc;
}

int pkv_bm_decode_step(pkv_bm* m, const int64_t* seq_ids, const int32_t* tokens, int n, int32_t* slot_mapping,
                       int32_t* context_lens, int32_t* block_tables, int max_blocks_per_seq, int32_t pad_value,
                       int32_t* cow_pairs) {
  if (!m) return -PKV_ERR_INVALID_ARG;
  std::lock_guard<std::mutex> lock(m->mu);
  if (n < 0 || max_blocks_per_seq < 0) return -PKV_ERR_INVALID_ARG;
  if (n == 0) return 0;
  if (!seq_ids || !tokens || !slot_mapping || !context_lens || !cow_pairs ||
      (!block_tables && max_blocks_per_seq > 0))
    return -PKV_ERR_INVALID_ARG;
  const int B = m->block_size;
  // Check the whole batch first, so that it either happens entirely or not
  // at all: known, distinct, resident sequences whose tables fit the row
  // width after the append, and enough blocks.  A shared tail is copied by
  // the first of its holders that appends; a later holder finds one
  // reference fewer, so the references each tail loses are counted as the
  // batch would drop them.
  std::vector<Sequence*> seqs(static_cast<size_t>(n));
  std::unordered_set<int64_t> seen;
  std::unordered_map<int, int> dropped;  // tail block -> references the batch drops before this point
  int need = 0;
  for (int i = 0; i < n; ++i) {
    const auto it = m->seqs.find(seq_ids[i]);
    if (it == m->seqs.end() || it->second.swapped || !seen.insert(seq_ids[i]).second) return -PKV_ERR_INVALID_ARG;
    Sequence& s = it->second;
    const int pos = static_cast<int>(s.tokens.size());
    if (pos / B + 1 > max_blocks_per_seq) return -PKV_ERR_INVALID_ARG;
    if (pos % B == 0) {
      ++need;
    } else {
      const int tail = s.table[pos / B];
      int& d = dropped[tail];
      if (m->blocks[tail].ref - d > 1) {
        ++need;
        ++d;
      }
    }
    seqs[static_cast<size_t>(i)] = &s;
  }
  if (need > available(m)) {
    ++m->refusals;
    return -PKV_ERR_OUT_OF_BLOCKS;
  }
  int pairs = 0;
  for (int i = 0; i < n; ++i) {
    int32_t src, dst;
    // cannot fail: the blocks were counted above
    append_locked(m, *seqs[static_cast<size_t>(i)], tokens[i], slot_mapping + i, &src, &dst);
    if (src >= 0) {
      cow_pairs[2 * pairs] = src;
      cow_pairs[2 * pairs + 1] = dst;
      ++pairs;
    }
  }
  for (int i = 0; i < n; ++i) {
    const Sequence& s = *seqs[static_cast<size_t>(i)];
    context_lens[i] = static_cast<int32_t>(s.tokens.size());
    int32_t* row = block_tables + static_cast<int64_t>(i) * max_blocks_per_seq;
    const int w = static_cast<int>(s.table.size());
    for (int j = 0; j < max_blocks_per_seq; ++j) row[j] = j < w ? s.table[j] : pad_value;
  }
  return pairs;
}

int pkv_bm_free_sequence(pkv_bm* m, int64_t seq_id) {
  if (!m) return -PKV_ERR_INVALID_ARG;
  std::lock_guard<std::mutex> lock(m->mu);
  const auto it = m->seqs.find(seq_id);
  if (it == m->seqs.end()) return -PKV_ERR_INVALID_ARG;
  if (!it->second.swapped)
    for (auto b = it->second.table.rbegin(); b != it->second.table.rend(); ++b) drop_ref(m, *b);
  m->seqs.erase(it);
  return PKV_OK;
}

int pkv_bm_seq_len(pkv_bm* m, int64_t seq_id) {
  if (!m) return -PKV_ERR_INVALID_ARG;
  std::lock_guard<std::mutex> lock(m->mu);
  const auto it = m->seqs.find(seq_id);
  return it == m->seqs.end() ? -PKV_ERR_INVALID_ARG : static_cast<int>(it->second.tokens.size());
}

int pkv_bm_seq_tokens(pkv_bm* m, int64_t seq_id, int32_t* out, int capacity) {
  if (!m) return -PKV_ERR_INVALID_ARG;
  std::lock_guard<std::mutex> lock(m->mu);
  const auto it = m->seqs.find(seq_id);
  if (it == m->seqs.end()) return -PKV_ERR_INVALID_ARG;
  const std::vector<int32_t>& t = it->second.tokens;
  const int n = static_cast<int>(t.size());
  if (n > capacity || (n > 0 && !out)) return -PKV_ERR_INVALID_ARG;
  if (n > 0) std::memcpy(out, t.data(), sizeof(int32_t) * static_cast<size_t>(n));
  return n;
}

int pkv_bm_block_table(pkv_bm* m, int64_t seq_id, int32_t* out, int capacity) {
  if (!m) return -PKV_ERR_INVALID_ARG;
  std::lock_guard<std::mutex> lock(m->mu);
  const auto it = m->seqs.find(seq_id);
  if (it == m->seqs.end() || it->second.swapped) return -PKV_ERR_INVALID_ARG;
  const int n = static_cast<int>(it->second.table.size());
  if (n > capacity || (n > 0 && !out)) return -PKV_ERR_INVALID_ARG;
  for (int i = 0; i < n; ++i) out[i] = it->second.table[i];
  return n;
}

int pkv_bm_swap_out(pkv_bm* m, int64_t seq_id, int32_t* blocks, int capacity) {
  if (!m) return -PKV_ERR_INVALID_ARG;
  std::lock_guard<std::mutex> lock(m->mu);
  const auto it = m->seqs.find(seq_id);
  if (it == m->seqs.end() || it->second.swapped) return -PKV_ERR_INVALID_ARG;
  Sequence& s = it->second;
  const int n = static_cast<int>(s.table.size());
  if (n > capacity || (n > 0 && !blocks)) return -PKV_ERR_INVALID_ARG;
  for (int i = 0; i < n; ++i) blocks[i] = s.table[i];
  for (int i = n - 1; i >= 0; --i) drop_ref(m, s.table[i]);
  s.table.clear();
  s.swapped = true;
  ++m->swap_outs;
  return n;
}

int pkv_bm_swap_in(pkv_bm* m, int64_t seq_id, int32_t* blocks, int capacity) {
  if (!m) return -PKV_ERR_INVALID_ARG;
  std::lock_guard<std::mutex> lock(m->mu);
  const auto it = m->seqs.find(seq_id);
  if (it == m->seqs.end() || !it->second.swapped) return -PKV_ERR_INVALID_ARG;
  Sequence& s = it->second;
  const int B = m->block_size;
  const int n = (static_cast<int>(s.tokens.size()) + B - 1) / B;
  if (n > capacity || (n > 0 && !blocks)) return -PKV_ERR_INVALID_ARG;
  if (n > available(m) - m->watermark) {  // resuming is an admission
    ++m->refusals;
    return -PKV_ERR_OUT_OF_BLOCKS;
  }
  for (int i = 0; i < n; ++i) {
    blocks[i] = take_block(m);
    s.table.push_back(blocks[i]);
  }
  s.swapped = false;
  for (int i = 0; (i + 1) * B <= static_cast<int>(s.tokens.size()); ++i) register_full(m, s, i);
  return n;
}

int pkv_bm_swap_in_cached(pkv_bm* m, int64_t seq_id, int32_t* blocks, int32_t* from_host, int capacity) {
  if (!m) return -PKV_ERR_INVALID_ARG;
  std::lock_guard<std::mutex> lock(m->mu);
  const auto it = m->seqs.find(seq_id);
  if (it == m->seqs.end() || !it->second.swapped) return -PKV_ERR_INVALID_ARG;
  Sequence& s = it->second;
  const int B = m->block_size;
  const int len = static_cast<int>(s.tokens.size());
  const int n = (len + B - 1) / B;
  if (n > capacity || (n > 0 && (!blocks || !from_host))) return -PKV_ERR_INVALID_ARG;
  // Full blocks from position 0 whose contents are still cached (the
  // admission rule: chained hash and tokens, up to the first miss).
  std::vector<int> hits;
  for (int i = 0; (i + 1) * B <= len; ++i) {
    const uint64_t parent = i == 0 ? s.root : s.hashes[static_cast<size_t>(i) - 1];
    const int b = lookup(m, s.hashes[static_cast<size_t>(i)], parent, s.tokens.data() + static_cast<size_t>(i) * B);
    if (b < 0) break;
    hits.push_back(b);
  }
  const int need = n - static_cast<int>(hits.size());
  int hit_evictable = 0;
  for (int b : hits) hit_evictable += m->blocks[b].ref == 0 ? 1 : 0;
  if (need > available(m) - hit_evictable - m->watermark) {  // resuming is an admission
    ++m->refusals;
    return -PKV_ERR_OUT_OF_BLOCKS;
  }
  for (size_t i = 0; i < hits.size(); ++i) {
    add_ref(m, hits[i]);
    s.table.push_back(hits[i]);
  }
  while (static_cast<int>(s.table.size()) < n) s.table.push_back(take_block(m));
  for (int i = 0; i < n; ++i) {
    blocks[i] = s.table[static_cast<size_t>(i)];
    from_host[i] = i < static_cast<int>(hits.size()) ? 0 : 1;
  }
  s.swapped = false;
  for (int i = static_cast<int>(hits.size()); (i + 1) * B <= len; ++i) register_full(m, s, i);
  return n;
}

int pkv_bm_get_stats(pkv_bm* m, pkv_bm_stats* out) {
  if (!m || !out) return -PKV_ERR_INVALID_ARG;
  std::lock_guard<std::mutex> lock(m->mu);
  const int B = m->block_size;
  pkv_bm_stats st{};
  st.num_blocks = m->num_blocks;
  st.block_size = B;
  st.blocks_free = static_cast<int64_t>(m->free_list.size());
  st.blocks_cached_unreferenced = static_cast<int64_t>(m->evictable.size());
  st.blocks_referenced = m->num_blocks - st.blocks_free - st.blocks_cached_unreferenced;
  st.blocks_cached = static_cast<int64_t>(m->cache.size());
  // Slots holding a token: per referenced block, the fill of its fullest
  // holder (holders of a shared block agree on the rows they share).
  std::vector<int> fill(static_cast<size_t>(m->num_blocks), 0);
  for (const auto& kv : m->seqs) {
    const pkv::Sequence& s = kv.second;
    if (s.swapped) {
      ++st.sequences_swapped;
      continue;
    }
    ++st.sequences_resident;
    const int len = static_cast<int>(s.tokens.size());
    const int nb = static_cast<int>(s.table.size());
    st.table_entries += nb;
    if (nb > st.max_blocks_per_sequence) st.max_blocks_per_sequence = nb;
    for (int j = 0; j < nb; ++j) {
      const int f = std::min(B, len - j * B);
      int& slot_fill = fill[static_cast<size_t>(s.table[static_cast<size_t>(j)])];
      if (f > slot_fill) slot_fill = f;
    }
  }
  for (int f : fill) st.slots_holding_tokens += f;
  st.prompt_tokens = m->prompt_tokens;
  st.prompt_tokens_cached = m->prompt_tokens_cached;
  st.evictions = m->evictions;
  st.cow_copies = m->cow_copies;
  st.swap_outs = m->swap_outs;
  st.refusals = m->refusals;
  *out = st;
  return PKV_OK;
}

}  // extern "C"
