// Host block manager for the paged KV cache.
//
// "KV Cache 与 vLLM" (zwxr.cn) §3.1-§3.4 and "KV Cache优化实战" §4.2: fixed
// 16-token physical blocks taken on demand, a per-sequence block table,
// prefix blocks shared by reference count and copied on write, blocks of a
// finished sequence returned at once.  The free list is a FIFO so the
// block a request gets is a deterministic function of the call history.
// Every mutating call validates first and changes nothing on error; an
// append batch is all-or-nothing (out of blocks must not crash a request:
// "企业官网建设流程全解析" §6.4).
//
// Optional prefix caching ("KV Cache优化实战" §5.2, "企业官网建设流程全解析"
// §6.2-§6.3): full blocks are registered under a hash chain of their token
// ids and a config key; a new request maps the longest chain of exact hits
// instead of recomputing it; a registered block whose references drop to
// zero stays cached and counts as free capacity, and is evicted only once
// the FIFO free list is empty -- leaves of the hash chain only (least
// recently used, then deepest, then lowest id), so no cached block loses the
// blocks it depends on.
#include <array>
#include <cstring>
#include <deque>
#include <set>
#include <string>
#include <tuple>
#include <unordered_map>
#include <vector>

#include "pkv.h"
#include "status.h"

struct pkv_bm {
  struct Seq {
    std::vector<int32_t> blocks;
    int32_t len = 0;
  };
  int32_t num_blocks = 0;
  int32_t block_size = PKV_BLOCK_SIZE;
  std::deque<int32_t> free_list;
  std::vector<int32_t> ref;
  std::unordered_map<int64_t, Seq> seqs;

  // ---- prefix cache ----
  using Key = std::tuple<uint64_t, int32_t, int32_t>;  // (last use, -depth, block): eviction order
  bool cache_on = false;
  uint64_t config_key = 0;
  uint64_t tick = 0;  // one per admit / commit / release call
  std::unordered_map<uint64_t, int32_t> by_hash;
  std::vector<uint8_t> reg;  // registered?
  std::vector<uint64_t> reg_hash;
  std::vector<int32_t> reg_parent, reg_depth, children;
  std::vector<std::array<int32_t, PKV_BLOCK_SIZE>> reg_tokens;
  std::vector<uint64_t> last_use;
  std::set<Key> leaves;     // registered, unreferenced, no registered child
  int32_t evictable = 0;    // registered, unreferenced
  int64_t lookups = 0, hits = 0, evictions = 0, registered = 0;

  Key key(int32_t b) const { return Key(last_use[b], -reg_depth[b], b); }
  bool is_leaf(int32_t b) const { return reg[b] && ref[b] == 0 && children[b] == 0; }
  int64_t available() const { return static_cast<int64_t>(free_list.size()) + evictable; }

  int32_t pop() {  // callers have checked available() > 0
    int32_t b;
    if (!free_list.empty()) {
      b = free_list.front();
      free_list.pop_front();
    } else {
      b = std::get<2>(*leaves.begin());
      unregister(b);
    }
    ref[b] = 1;
    return b;
  }
  void unregister(int32_t b) {  // b is an evictable leaf
    leaves.erase(key(b));
    by_hash.erase(reg_hash[b]);
    reg[b] = 0;
    --evictable;
    --registered;
    ++evictions;
    const int32_t p = reg_parent[b];
    if (p >= 0 && --children[p] == 0 && is_leaf(p)) leaves.insert(key(p));
  }
  void drop(int32_t b) {
    if (--ref[b] != 0) return;
    if (!cache_on || !reg[b]) {
      free_list.push_back(b);
      return;
    }
    last_use[b] = tick;
    ++evictable;
    if (children[b] == 0) leaves.insert(key(b));
  }
  void take(int32_t b) {  // a cache hit adds a reference
    if (ref[b] == 0) {
      --evictable;
      if (children[b] == 0) leaves.erase(key(b));
    }
    ++ref[b];
    last_use[b] = tick;
  }
};

namespace {

// FNV-1a 64-bit (Fowler-Noll-Vo; offset basis 0xcbf29ce484222325, prime
// 0x100000001b3) over the given bytes, continuing from h.
uint64_t fnv1a(uint64_t h, const uint8_t *data, size_t n) {
  for (size_t i = 0; i < n; ++i) {
    h ^= data[i];
    h *= 0x100000001b3ull;
  }
  return h;
}

void put_le(uint8_t *dst, uint64_t v, int bytes) {
  for (int i = 0; i < bytes; ++i) dst[i] = static_cast<uint8_t>(v >> (8 * i));
}

}  // namespace

using pkv::fail;

extern "C" {

pkv_status pkv_bm_create(int32_t num_blocks, int32_t block_size, const int32_t *alloc_order,
                         pkv_bm **out) {
  if (!out) return fail(PKV_ERR_INVALID, "pkv_bm_create: out is NULL");
  if (num_blocks <= 0) return fail(PKV_ERR_INVALID, "pkv_bm_create: num_blocks must be > 0");
  if (block_size != PKV_BLOCK_SIZE && block_size != PKV_BLOCK_SIZE_32)
    return fail(PKV_ERR_UNSUPPORTED, "pkv_bm_create: block_size must be 16 or 32");
  std::vector<char> seen(num_blocks, 0);
  if (alloc_order) {
    for (int32_t i = 0; i < num_blocks; ++i) {
      int32_t b = alloc_order[i];
      if (b < 0 || b >= num_blocks || seen[b])
        return fail(PKV_ERR_INVALID, "pkv_bm_create: alloc_order is not a permutation");
      seen[b] = 1;
    }
  }
  pkv_bm *bm = new pkv_bm();
  bm->num_blocks = num_blocks;
  bm->block_size = block_size;
  bm->ref.assign(num_blocks, 0);
  for (int32_t i = 0; i < num_blocks; ++i) bm->free_list.push_back(alloc_order ? alloc_order[i] : i);
  *out = bm;
  return PKV_OK;
}

void pkv_bm_destroy(pkv_bm *bm) { delete bm; }

pkv_status kv_block_alloc(pkv_bm *bm, int32_t *block_id) {
  if (!bm || !block_id) return fail(PKV_ERR_INVALID, "kv_block_alloc: NULL argument");
  if (bm->available() == 0) return fail(PKV_ERR_NO_BLOCKS, "kv_block_alloc: no free or evictable block");
  *block_id = bm->pop();
  return PKV_OK;
}

pkv_status kv_block_free(pkv_bm *bm, int32_t block_id) {
  if (!bm) return fail(PKV_ERR_INVALID, "kv_block_free: NULL handle");
  if (block_id < 0 || block_id >= bm->num_blocks || bm->ref[block_id] <= 0)
    return fail(PKV_ERR_INVALID, "kv_block_free: block is not held");
  ++bm->tick;
  bm->drop(block_id);
  return PKV_OK;
}

pkv_status pkv_seq_create(pkv_bm *bm, int64_t seq_id) {
  if (!bm) return fail(PKV_ERR_INVALID, "pkv_seq_create: NULL handle");
  if (bm->seqs.count(seq_id)) return fail(PKV_ERR_INVALID, "pkv_seq_create: sequence exists");
  bm->seqs.emplace(seq_id, pkv_bm::Seq());
  return PKV_OK;
}

pkv_status pkv_seq_fork(pkv_bm *bm, int64_t parent, int64_t child) {
  if (!bm) return fail(PKV_ERR_INVALID, "pkv_seq_fork: NULL handle");
  auto it = bm->seqs.find(parent);
  if (it == bm->seqs.end()) return fail(PKV_ERR_INVALID, "pkv_seq_fork: unknown parent");
  if (bm->seqs.count(child)) return fail(PKV_ERR_INVALID, "pkv_seq_fork: child exists");
  pkv_bm::Seq s = it->second;
  for (int32_t b : s.blocks) ++bm->ref[b];
  bm->seqs.emplace(child, std::move(s));
  return PKV_OK;
}

pkv_status pkv_seq_free(pkv_bm *bm, int64_t seq_id) {
  if (!bm) return fail(PKV_ERR_INVALID, "pkv_seq_free: NULL handle");
  auto it = bm->seqs.find(seq_id);
  if (it == bm->seqs.end()) return fail(PKV_ERR_INVALID, "pkv_seq_free: unknown sequence");
  ++bm->tick;
  for (int32_t b : it->second.blocks) bm->drop(b);
  bm->seqs.erase(it);
  return PKV_OK;
}

pkv_status pkv_seq_append_slots(pkv_bm *bm, const int64_t *seq_ids, int32_t n,
                                int32_t *slot_mapping, int32_t *cow_src, int32_t *cow_dst,
                                int32_t *num_cow) {
  if (!bm || n < 0 || (n > 0 && (!seq_ids || !slot_mapping || !cow_src || !cow_dst)) || !num_cow)
    return fail(PKV_ERR_INVALID, "pkv_seq_append_slots: bad argument");
  const int32_t bs = bm->block_size;
  // Dry run: count the blocks the batch takes, tracking lengths, which last
  // blocks are already private to the appender, and reference drops.
  struct Local {
    int32_t len;
    bool last_private;  // last block was taken in this batch (count 1, exclusive)
  };
  std::unordered_map<int64_t, Local> local;
  std::unordered_map<int32_t, int32_t> ref_drop;
  int64_t need = 0;
  for (int32_t i = 0; i < n; ++i) {
    auto it = bm->seqs.find(seq_ids[i]);
    if (it == bm->seqs.end()) return fail(PKV_ERR_INVALID, "pkv_seq_append_slots: unknown sequence");
    auto ins = local.emplace(seq_ids[i], Local{it->second.len, false});
    Local &l = ins.first->second;
    if (l.len % bs == 0) {
      ++need;
      l.last_private = true;
    } else if (!l.last_private) {
      int32_t last = it->second.blocks.back();
      if (bm->ref[last] - ref_drop[last] > 1) {
        ++need;
        ++ref_drop[last];
      }
      l.last_private = true;  // after a copy, or when this holder is the last one
    }
    if (l.len == INT32_MAX) return fail(PKV_ERR_INVALID, "pkv_seq_append_slots: length overflow");
    ++l.len;
  }
  if (need > bm->available())
    return fail(PKV_ERR_NO_BLOCKS, "pkv_seq_append_slots: free and evictable blocks cannot cover the batch");
  // Apply.
  int32_t ncow = 0;
  for (int32_t i = 0; i < n; ++i) {
    pkv_bm::Seq &s = bm->seqs[seq_ids[i]];
    int32_t pos = s.len;
    if (pos % bs == 0) {
      s.blocks.push_back(bm->pop());
    } else {
      int32_t last = s.blocks.back();
      if (bm->ref[last] > 1) {
        int32_t fresh = bm->pop();
        --bm->ref[last];
        s.blocks.back() = fresh;
        cow_src[ncow] = last;
        cow_dst[ncow] = fresh;
        ++ncow;
      }
    }
    slot_mapping[i] = s.blocks[pos / bs] * bs + pos % bs;
    s.len = pos + 1;
  }
  *num_cow = ncow;
  return PKV_OK;
}

pkv_status pkv_build_block_tables(const pkv_bm *bm, const int64_t *seq_ids, int32_t n,
                                  int32_t max_blocks, int32_t *tables, int32_t *context_lens) {
  if (!bm || n < 0 || max_blocks < 0 || (n > 0 && (!seq_ids || !context_lens)) ||
      (n > 0 && max_blocks > 0 && !tables))
    return fail(PKV_ERR_INVALID, "pkv_build_block_tables: bad argument");
  for (int32_t i = 0; i < n; ++i) {
    auto it = bm->seqs.find(seq_ids[i]);
    if (it == bm->seqs.end()) return fail(PKV_ERR_INVALID, "pkv_build_block_tables: unknown sequence");
    if (static_cast<int64_t>(it->second.blocks.size()) > max_blocks)
      return fail(PKV_ERR_INVALID, "pkv_build_block_tables: table longer than max_blocks");
  }
  for (int32_t i = 0; i < n; ++i) {
    const pkv_bm::Seq &s = bm->seqs.at(seq_ids[i]);
    int32_t *row = tables + static_cast<int64_t>(i) * max_blocks;
    int32_t nb = static_cast<int32_t>(s.blocks.size());
    for (int32_t j = 0; j < nb; ++j) row[j] = s.blocks[j];
    for (int32_t j = nb; j < max_blocks; ++j) row[j] = -1;
    context_lens[i] = s.len;
  }
  return PKV_OK;
}

int32_t pkv_bm_num_free(const pkv_bm *bm) {
  return bm ? static_cast<int32_t>(bm->available()) : -1;
}

int32_t pkv_bm_num_blocks(const pkv_bm *bm) { return bm ? bm->num_blocks : -1; }

int32_t pkv_bm_block_size(const pkv_bm *bm) { return bm ? bm->block_size : -1; }

pkv_status pkv_bm_free_list(const pkv_bm *bm, int32_t *out, int32_t cap, int32_t *n) {
  if (!bm || !n || cap < 0 || (cap > 0 && !out))
    return fail(PKV_ERR_INVALID, "pkv_bm_free_list: bad argument");
  int32_t i = 0;
  for (int32_t b : bm->free_list) {
    if (i >= cap) break;
    out[i++] = b;
  }
  *n = static_cast<int32_t>(bm->free_list.size());
  return PKV_OK;
}

pkv_status pkv_bm_refcount(const pkv_bm *bm, int32_t block_id, int32_t *count) {
  if (!bm || !count || block_id < 0 || block_id >= bm->num_blocks)
    return fail(PKV_ERR_INVALID, "pkv_bm_refcount: bad argument");
  *count = bm->ref[block_id];
  return PKV_OK;
}

pkv_status pkv_seq_len(const pkv_bm *bm, int64_t seq_id, int32_t *len) {
  if (!bm || !len) return fail(PKV_ERR_INVALID, "pkv_seq_len: bad argument");
  auto it = bm->seqs.find(seq_id);
  if (it == bm->seqs.end()) return fail(PKV_ERR_INVALID, "pkv_seq_len: unknown sequence");
  *len = it->second.len;
  return PKV_OK;
}

// K plus V bytes of one token for one KV head (codes' scales included).
static int64_t kv_bytes_per_token_head(int32_t head_dim, pkv_dtype dt) {
  const int64_t d = head_dim;
  switch (dt) {
    case PKV_F16:
    case PKV_BF16:
      return 2 * (2 * d);
    case PKV_FP8_E4M3:
    case PKV_FP8_E5M2:
    case PKV_INT8:
      return 2 * (d + 4);  // codes + one fp32 scale, K and V
    case PKV_FP8_E4M3_INT4:
      return (d + 4) + (d / 2 + 4);  // one-byte K codes, 4-bit V codes, a scale each
    default:
      return -1;  // not a cache type
  }
}

int64_t pkv_kv_bytes(int32_t layers, int32_t kv_heads, int32_t head_dim, int64_t tokens,
                     pkv_dtype cache_dtype) {
  int64_t per = kv_bytes_per_token_head(head_dim, cache_dtype);
  if (layers < 0 || kv_heads < 0 || head_dim <= 0 || (head_dim & 1) || tokens < 0 || per < 0) return -1;
  return static_cast<int64_t>(layers) * kv_heads * tokens * per;
}

int64_t pkv_pool_blocks(int64_t budget_bytes, int32_t layers, int32_t kv_heads, int32_t head_dim,
                        pkv_dtype cache_dtype, int32_t block_size) {
  if (block_size != PKV_BLOCK_SIZE && block_size != PKV_BLOCK_SIZE_32) return -1;
  int64_t per_block = pkv_kv_bytes(layers, kv_heads, head_dim, block_size, cache_dtype);
  if (budget_bytes < 0 || per_block <= 0) return -1;
  return budget_bytes / per_block;
}

// ---- prefix cache -------------------------------------------------------------

uint64_t pkv_block_hash(uint64_t parent_hash, const int32_t *tokens, uint64_t config_key) {
  uint8_t buf[8 + 4 * PKV_BLOCK_SIZE + 8];
  put_le(buf, parent_hash, 8);
  for (int i = 0; i < PKV_BLOCK_SIZE; ++i) put_le(buf + 8 + 4 * i, static_cast<uint32_t>(tokens[i]), 4);
  put_le(buf + 8 + 4 * PKV_BLOCK_SIZE, config_key, 8);
  return fnv1a(0xcbf29ce484222325ull, buf, sizeof(buf));
}

pkv_status pkv_bm_enable_prefix_cache(pkv_bm *bm, uint64_t config_key) {
  if (!bm) return fail(PKV_ERR_INVALID, "pkv_bm_enable_prefix_cache: NULL handle");
  if (bm->cache_on) return fail(PKV_ERR_INVALID, "pkv_bm_enable_prefix_cache: already enabled");
  if (bm->block_size != PKV_BLOCK_SIZE)
    return fail(PKV_ERR_UNSUPPORTED, "pkv_bm_enable_prefix_cache: needs 16-token blocks");
  const size_t n = static_cast<size_t>(bm->num_blocks);
  bm->cache_on = true;
  bm->config_key = config_key;
  bm->reg.assign(n, 0);
  bm->reg_hash.assign(n, 0);
  bm->reg_parent.assign(n, -1);
  bm->reg_depth.assign(n, 0);
  bm->children.assign(n, 0);
  bm->reg_tokens.assign(n, {});
  bm->last_use.assign(n, 0);
  return PKV_OK;
}

pkv_status pkv_seq_admit(pkv_bm *bm, int64_t seq_id, const int32_t *tokens, int32_t num_tokens,
                         int32_t *num_cached) {
  if (!bm || !num_cached || num_tokens < 0 || (num_tokens > 0 && !tokens))
    return fail(PKV_ERR_INVALID, "pkv_seq_admit: bad argument");
  if (!bm->cache_on) return fail(PKV_ERR_INVALID, "pkv_seq_admit: prefix cache not enabled");
  if (bm->seqs.count(seq_id)) return fail(PKV_ERR_INVALID, "pkv_seq_admit: sequence exists");
  ++bm->tick;
  pkv_bm::Seq seq;
  const int32_t bs = bm->block_size;
  const int32_t usable = num_tokens > 0 ? (num_tokens - 1) / bs : 0;  // at least one token is computed
  uint64_t h = 0;
  int32_t parent = -1;
  for (int32_t j = 0; j < usable; ++j) {
    const int32_t *blk = tokens + static_cast<int64_t>(j) * bs;
    h = pkv_block_hash(h, blk, bm->config_key);
    ++bm->lookups;
    auto it = bm->by_hash.find(h);
    if (it == bm->by_hash.end()) break;
    const int32_t b = it->second;
    if (bm->reg_parent[b] != parent || std::memcmp(bm->reg_tokens[b].data(), blk, sizeof(int32_t) * bs) != 0)
      break;  // a hash collision or a stale chain: treat as a miss
    ++bm->hits;
    bm->take(b);
    seq.blocks.push_back(b);
    parent = b;
  }
  seq.len = static_cast<int32_t>(seq.blocks.size()) * bs;
  *num_cached = seq.len;
  bm->seqs.emplace(seq_id, std::move(seq));
  return PKV_OK;
}

pkv_status pkv_seq_commit_prefix(pkv_bm *bm, int64_t seq_id, const int32_t *tokens, int32_t num_tokens,
                                 int32_t *num_registered) {
  if (!bm || num_tokens < 0 || (num_tokens > 0 && !tokens))
    return fail(PKV_ERR_INVALID, "pkv_seq_commit_prefix: bad argument");
  if (!bm->cache_on) return fail(PKV_ERR_INVALID, "pkv_seq_commit_prefix: prefix cache not enabled");
  auto it = bm->seqs.find(seq_id);
  if (it == bm->seqs.end()) return fail(PKV_ERR_INVALID, "pkv_seq_commit_prefix: unknown sequence");
  if (num_tokens > it->second.len)
    return fail(PKV_ERR_INVALID, "pkv_seq_commit_prefix: more tokens than the sequence holds");
  ++bm->tick;
  const int32_t bs = bm->block_size;
  const std::vector<int32_t> &blocks = it->second.blocks;
  uint64_t h = 0;
  int32_t parent = -1, added = 0;
  for (int32_t j = 0; j < num_tokens / bs; ++j) {
    const int32_t *blk = tokens + static_cast<int64_t>(j) * bs;
    h = pkv_block_hash(h, blk, bm->config_key);
    const int32_t b = blocks[j];
    auto hit = bm->by_hash.find(h);
    if (hit != bm->by_hash.end()) {
      if (hit->second != b) break;  // a duplicate of another block: this sequence's chain stops
    } else if (!bm->reg[b]) {
      bm->by_hash.emplace(h, b);
      bm->reg[b] = 1;
      bm->reg_hash[b] = h;
      bm->reg_parent[b] = parent;
      bm->reg_depth[b] = j;
      std::memcpy(bm->reg_tokens[b].data(), blk, sizeof(int32_t) * bs);
      bm->last_use[b] = bm->tick;
      if (parent >= 0) {
        if (bm->is_leaf(parent)) bm->leaves.erase(bm->key(parent));
        ++bm->children[parent];
      }
      ++bm->registered;
      ++added;
    } else {
      break;  // b is registered under another chain: this sequence's chain stops
    }
    parent = b;
  }
  if (num_registered) *num_registered = added;
  return PKV_OK;
}

pkv_status pkv_prefix_cache_stats(const pkv_bm *bm, pkv_prefix_stats *out) {
  if (!bm || !out) return fail(PKV_ERR_INVALID, "pkv_prefix_cache_stats: NULL argument");
  out->lookups = bm->lookups;
  out->hits = bm->hits;
  out->evictions = bm->evictions;
  out->registered = bm->registered;
  out->evictable = bm->evictable;
  return PKV_OK;
}

}  // extern "C"
