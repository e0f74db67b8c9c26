// Host block manager of libpagedkv: free list, block tables, reference
// counts, fork and block-granular copy-on-write.
//
// Semantics ("Paged KV Cache Allocation and the Block Table", the
// append_token routine and "Sharing blocks between sequences"; "PagedAttention"
// S06, the BlockManager listing, "Copy-on-write, for free" and "Reference
// counts must be exact"; "paged attention deep", "Copy-on-write for shared
// prefixes"):
//   * Appending token t to a sequence of length L: when L is a multiple of B
//     the table grows by one block popped from the free list; otherwise, if
//     the partly filled tail block is named by more than one table, the
//     sequence swaps it for a fresh private block (the caller copies the
//     contents with pk_copy_blocks) and the shared block loses one
//     reference. The slot is table[L / B] * B + L % B.
//   * Fork: the child names the parent's blocks; each count goes up by one.
//   * Retire: each block of the table loses one reference; those reaching
//     zero go back to the free list, in table order.
//   * The free list is a stack whose first pop is alloc_order[0].
//   * Prefix caching ("PagedAttention" S06, "What's next": block contents are
//     hashed so that requests with a common prefix share physical blocks):
//     a full block is registered under a 64-bit hash chained over every token
//     up to and including it, and verified on lookup against its depth, its
//     parent's chain hash and its own tokens. A cached block whose last
//     reference goes away stays cached; allocations take the free list first
//     and then evict the unreferenced cached block released longest ago,
//     deepest first among blocks released by one call.
// Appends are all or nothing (a batch counts the blocks it needs first).
#include <algorithm>
#include <cstdint>
#include <cstring>
#include <new>
#include <set>
#include <tuple>
#include <unordered_map>
#include <vector>

#include "pagedkv.h"

namespace {

struct Sequence {
  int64_t len = 0;
  std::vector<int32_t> table;  // device block ids, or host block ids when swapped
  bool swapped = false;
  uint64_t batch_mark = 0;     // batch call that last counted this sequence
  int64_t batch_grown = 0;     // tokens that call counted for it so far
};

// Room for `blocks` table entries, growing geometrically (an exact reserve
// would reallocate the table every time it gains a block).
inline void reserve_table(std::vector<int32_t> &t, int64_t blocks) {
  if (int64_t(t.capacity()) < blocks)
    t.reserve(size_t(std::max<int64_t>(blocks, 2 * int64_t(t.capacity()))));
}

// Prefix-cache entry of one block.
struct CacheEntry {
  bool cached = false;
  int32_t depth = 0;             // block index in every table that names it
  uint64_t chain = 0;            // hash of tokens [0, (depth + 1) * B)
  uint64_t parent = 0;           // hash of tokens [0, depth * B)
  std::vector<int32_t> tokens;   // the block's own B tokens
  int64_t released = 0;          // clock of the call that left it unreferenced
};

// Chained block hash: the SplitMix64 output function (Steele, Lea and Flood,
// "Fast splittable pseudorandom number generators", 2014) applied after each
// token is added in.
inline uint64_t mix64(uint64_t z) {
  z = (z ^ (z >> 30)) * 0xbf58476d1ce4e5b9ull;
  z = (z ^ (z >> 27)) * 0x94d049bb133111ebull;
  return z ^ (z >> 31);
}

inline uint64_t chain_hash(uint64_t parent, const int32_t *tok, int32_t n) {
  uint64_t h = parent;
  for (int32_t i = 0; i < n; ++i) h = mix64(h + 0x9e3779b97f4a7c15ull + uint32_t(tok[i]));
  return h;
}

constexpr uint64_t kChainSeed = 0x243f6a8885a308d3ull;

// Unreferenced cached blocks in eviction order: oldest release first, then
// the deepest block, then the lowest id.
using EvictKey = std::tuple<int64_t, int32_t, int32_t>;

}  // namespace

struct pk_bm {
  int32_t num_blocks = 0;
  int32_t block_size = 0;
  std::vector<int32_t> free_stack;  // back() is handed out next
  std::vector<int32_t> refs;
  std::unordered_map<int64_t, Sequence> seqs;
  int64_t cow_copies = 0;
  int32_t num_host_blocks = 0;           // swap space in host memory
  std::vector<int32_t> host_free;        // back() is handed out next
  // prefix cache
  std::vector<CacheEntry> entry;                    // per block
  std::unordered_multimap<uint64_t, int32_t> index;  // chain hash -> cached block
  std::set<EvictKey> idle;                          // unreferenced cached blocks
  int64_t clock = 0;
  int64_t cache_hits = 0;
  int64_t evictions = 0;
  // batch pre-count: per-call marks instead of per-call maps
  uint64_t batch_epoch = 0;
  std::vector<uint64_t> given_up_mark;   // per block: call that last counted a CoW of it
  std::vector<int32_t> given_up;         // CoW copies of the block that call counted
  std::vector<Sequence *> batch_seqs;    // scratch of pk_bm_append_batch

  int64_t blocks_for(int64_t len) const { return (len + block_size - 1) / block_size; }

  // Blocks an allocation can take: the free list plus the idle cached blocks.
  int64_t available() const { return int64_t(free_stack.size()) + int64_t(idle.size()); }

  EvictKey idle_key(int32_t b) const { return EvictKey(entry[b].released, -entry[b].depth, b); }

  void uncache(int32_t b) {
    CacheEntry &e = entry[b];
    auto range = index.equal_range(e.chain);
    for (auto it = range.first; it != range.second; ++it)
      if (it->second == b) {
        index.erase(it);
        break;
      }
    e.cached = false;
    e.tokens.clear();
    e.tokens.shrink_to_fit();
  }

  // One block for a table (available() > 0 checked by the caller): the top
  // of the free list, else the first idle cached block, which leaves the cache.
  int32_t take_block() {
    if (!free_stack.empty()) {
      const int32_t b = free_stack.back();
      free_stack.pop_back();
      return b;
    }
    const int32_t b = std::get<2>(*idle.begin());
    idle.erase(idle.begin());
    uncache(b);
    ++evictions;
    return b;
  }

  // A table stops naming block b.
  void release(int32_t b) {
    if (--refs[b] != 0) return;
    if (entry[b].cached) {
      entry[b].released = clock;
      idle.insert(idle_key(b));
    } else {
      free_stack.push_back(b);
    }
  }

  // The cached block holding the prefix whose last block is tok[0, B) at
  // `depth`, after a prefix with chain hash `parent`; -1 if none.
  int32_t find_cached(uint64_t chain, uint64_t parent, int32_t depth, const int32_t *tok) const {
    auto range = index.equal_range(chain);
    for (auto it = range.first; it != range.second; ++it) {
      const CacheEntry &e = entry[it->second];
      if (e.depth == depth && e.parent == parent &&
          std::equal(e.tokens.begin(), e.tokens.end(), tok))
        return it->second;
    }
    return -1;
  }

  // Appends one token (the caller has checked that a block is available if
  // one is needed). A new block or a CoW copy comes from take_block.
  int64_t append_one(Sequence &s, int64_t *cow_src, int64_t *cow_dst) {
    const int64_t off = s.len % block_size;
    if (off == 0) {
      const int32_t b = take_block();
      refs[b] = 1;
      s.table.push_back(b);
    } else {
      const int32_t tail = s.table.back();
      if (refs[tail] > 1) {
        const int32_t b = take_block();
        refs[b] = 1;
        refs[tail] -= 1;
        s.table.back() = b;
        ++cow_copies;
        if (cow_src) *cow_src = tail;
        if (cow_dst) *cow_dst = b;
      }
    }
    const int64_t slot = int64_t(s.table[s.len / block_size]) * block_size + off;
    s.len += 1;
    return slot;
  }
};

extern "C" {

pk_status pk_bm_create(int32_t num_blocks, int32_t block_size, const int32_t *alloc_order,
                       pk_bm **out) {
  if (!out || num_blocks <= 0 || block_size <= 0) return PK_ERR_INVALID_ARG;
  *out = nullptr;
  pk_bm *bm = new (std::nothrow) pk_bm;
  if (!bm) return PK_ERR_NOMEM;
  try {
    bm->num_blocks = num_blocks;
    bm->block_size = block_size;
    bm->refs.assign(num_blocks, 0);
    bm->entry.resize(num_blocks);
    bm->given_up_mark.assign(num_blocks, 0);
    bm->given_up.assign(num_blocks, 0);
    bm->free_stack.resize(num_blocks);
    std::vector<char> seen(num_blocks, 0);
    for (int32_t i = 0; i < num_blocks; ++i) {
      const int32_t b = alloc_order ? alloc_order[i] : i;
      if (b < 0 || b >= num_blocks || seen[b]) {
        delete bm;
        return PK_ERR_INVALID_ARG;
      }
      seen[b] = 1;
      bm->free_stack[num_blocks - 1 - i] = b;  // alloc_order[0] ends on top
    }
  } catch (const std::bad_alloc &) {
    delete bm;
    return PK_ERR_NOMEM;
  }
  *out = bm;
  return PK_OK;
}

void pk_bm_destroy(pk_bm *bm) { delete bm; }

pk_status pk_bm_add_seq(pk_bm *bm, int64_t seq_id) {
  if (!bm) return PK_ERR_INVALID_ARG;
  try {
    auto r = bm->seqs.emplace(seq_id, Sequence{});
    return r.second ? PK_OK : PK_ERR_SEQ_EXISTS;
  } catch (const std::bad_alloc &) {
    return PK_ERR_NOMEM;
  }
}

pk_status pk_bm_append_slots(pk_bm *bm, int64_t seq_id, int32_t n, int64_t *slots_out,
                             int64_t *cow_pairs_out, int32_t *n_cow_out) {
  if (!bm || n < 0 || (n > 0 && !slots_out)) return PK_ERR_INVALID_ARG;
  if (n_cow_out) *n_cow_out = 0;
  auto it = bm->seqs.find(seq_id);
  if (it == bm->seqs.end()) return PK_ERR_UNKNOWN_SEQ;
  Sequence &s = it->second;
  if (s.swapped) return PK_ERR_INVALID_ARG;
  if (n == 0) return PK_OK;
  // Blocks needed: one per block boundary crossed, plus a CoW copy when the
  // first token lands in a shared, partly filled tail.
  const int64_t fresh = bm->blocks_for(s.len + n) - bm->blocks_for(s.len);
  const int64_t cow = (s.len % bm->block_size != 0 && bm->refs[s.table.back()] > 1) ? 1 : 0;
  if (fresh + cow > bm->available()) return PK_ERR_OUT_OF_BLOCKS;
  try {
    reserve_table(s.table, bm->blocks_for(s.len + n));
  } catch (const std::bad_alloc &) {
    return PK_ERR_NOMEM;
  }
  int64_t src = -1, dst = -1;
  for (int32_t i = 0; i < n; ++i) slots_out[i] = bm->append_one(s, &src, &dst);
  if (src >= 0) {
    if (cow_pairs_out) {
      cow_pairs_out[0] = src;
      cow_pairs_out[1] = dst;
    }
    if (n_cow_out) *n_cow_out = 1;
  }
  return PK_OK;
}

pk_status pk_bm_append_batch(pk_bm *bm, const int64_t *seq_ids, int32_t n, int64_t *slots_out,
                             int64_t *cow_pairs_out, int32_t *n_cow_out) {
  if (!bm || n < 0 || (n > 0 && (!seq_ids || !slots_out))) return PK_ERR_INVALID_ARG;
  if (n_cow_out) *n_cow_out = 0;
  std::vector<Sequence *> &seqp = bm->batch_seqs;
  int64_t need = 0;
  try {
    seqp.clear();
    seqp.reserve(n);
    // Count the blocks the whole batch takes before changing anything: a
    // token at a block boundary takes one; a token landing in a tail another
    // table still names takes a CoW copy (siblings earlier in the batch may
    // already have given that tail up). A sequence's tail is private after
    // its first token of the batch.
    const uint64_t ep = ++bm->batch_epoch;
    for (int32_t i = 0; i < n; ++i) {
      auto it = bm->seqs.find(seq_ids[i]);
      if (it == bm->seqs.end()) return PK_ERR_UNKNOWN_SEQ;
      Sequence &s = it->second;
      if (s.swapped) return PK_ERR_INVALID_ARG;
      seqp.push_back(&s);
      if (s.batch_mark != ep) {
        s.batch_mark = ep;
        s.batch_grown = 0;
      }
      if ((s.len + s.batch_grown) % bm->block_size == 0) {
        ++need;
      } else if (s.batch_grown == 0) {
        const int32_t tail = s.table.back();
        if (bm->given_up_mark[tail] != ep) {
          bm->given_up_mark[tail] = ep;
          bm->given_up[tail] = 0;
        }
        if (bm->refs[tail] - bm->given_up[tail] > 1) {
          ++need;
          ++bm->given_up[tail];
        }
      }
      ++s.batch_grown;
      reserve_table(s.table, bm->blocks_for(s.len + s.batch_grown));
    }
  } catch (const std::bad_alloc &) {
    return PK_ERR_NOMEM;
  }
  if (need > bm->available()) return PK_ERR_OUT_OF_BLOCKS;
  int32_t ncow = 0;
  for (int32_t i = 0; i < n; ++i) {
    int64_t src = -1, dst = -1;
    slots_out[i] = bm->append_one(*seqp[i], &src, &dst);
    if (src >= 0) {
      if (cow_pairs_out) {
        cow_pairs_out[2 * ncow] = src;
        cow_pairs_out[2 * ncow + 1] = dst;
      }
      ++ncow;
    }
  }
  if (n_cow_out) *n_cow_out = ncow;
  return PK_OK;
}

pk_status pk_bm_fork(pk_bm *bm, int64_t parent, int64_t child) {
  if (!bm) return PK_ERR_INVALID_ARG;
  if (bm->seqs.count(child)) return PK_ERR_SEQ_EXISTS;
  auto it = bm->seqs.find(parent);
  if (it == bm->seqs.end()) return PK_ERR_UNKNOWN_SEQ;
  if (it->second.swapped) return PK_ERR_INVALID_ARG;
  try {
    Sequence copy = it->second;
    for (int32_t b : copy.table) bm->refs[b] += 1;
    bm->seqs.emplace(child, std::move(copy));
  } catch (const std::bad_alloc &) {
    return PK_ERR_NOMEM;
  }
  return PK_OK;
}

pk_status pk_bm_free_seq(pk_bm *bm, int64_t seq_id) {
  if (!bm) return PK_ERR_INVALID_ARG;
  auto it = bm->seqs.find(seq_id);
  if (it == bm->seqs.end()) return PK_ERR_UNKNOWN_SEQ;
  ++bm->clock;
  for (int32_t b : it->second.table) {
    if (it->second.swapped)
      bm->host_free.push_back(b);  // a swapped sequence holds host blocks
    else
      bm->release(b);
  }
  bm->seqs.erase(it);
  return PK_OK;
}

pk_status pk_bm_seq_len(const pk_bm *bm, int64_t seq_id, int64_t *len_out) {
  if (!bm || !len_out) return PK_ERR_INVALID_ARG;
  auto it = bm->seqs.find(seq_id);
  if (it == bm->seqs.end()) return PK_ERR_UNKNOWN_SEQ;
  *len_out = it->second.len;
  return PK_OK;
}

pk_status pk_bm_block_table(const pk_bm *bm, int64_t seq_id, int32_t *out, int32_t cap,
                            int32_t *len_out) {
  if (!bm || cap < 0 || (cap > 0 && !out)) return PK_ERR_INVALID_ARG;
  auto it = bm->seqs.find(seq_id);
  if (it == bm->seqs.end()) return PK_ERR_UNKNOWN_SEQ;
  const auto &t = it->second.table;
  const int32_t m = std::min<int32_t>(cap, int32_t(t.size()));
  if (m > 0) std::memcpy(out, t.data(), sizeof(int32_t) * size_t(m));
  if (len_out) *len_out = int32_t(t.size());
  return PK_OK;
}

pk_status pk_bm_export_tables(const pk_bm *bm, const int64_t *seq_ids, int32_t n,
                              int32_t max_blocks, int32_t *tables_out, int32_t *lens_out) {
  if (!bm || n < 0 || max_blocks < 0 || (n > 0 && (!seq_ids || !tables_out)))
    return PK_ERR_INVALID_ARG;
  for (int32_t i = 0; i < n; ++i) {
    auto it = bm->seqs.find(seq_ids[i]);
    if (it == bm->seqs.end()) return PK_ERR_UNKNOWN_SEQ;
    const auto &s = it->second;
    if (s.swapped || int64_t(s.table.size()) > max_blocks || s.len > INT32_MAX)
      return PK_ERR_INVALID_ARG;
    int32_t *row = tables_out + size_t(i) * size_t(max_blocks);
    std::copy(s.table.begin(), s.table.end(), row);
    std::fill(row + s.table.size(), row + max_blocks, -1);
    if (lens_out) lens_out[i] = int32_t(s.len);
  }
  return PK_OK;
}

int32_t pk_bm_num_free(const pk_bm *bm) { return bm ? int32_t(bm->available()) : -1; }

int32_t pk_bm_refcount(const pk_bm *bm, int32_t block) {
  if (!bm || block < 0 || block >= bm->num_blocks) return -1;
  return bm->refs[block];
}

pk_status pk_bm_check_invariants(const pk_bm *bm) {
  if (!bm) return PK_ERR_INVALID_ARG;
  std::vector<int32_t> count(bm->num_blocks, 0);
  std::vector<char> host_used(bm->num_host_blocks, 0);
  int64_t host_held = 0;
  for (const auto &kv : bm->seqs) {
    const Sequence &s = kv.second;
    if (int64_t(s.table.size()) != bm->blocks_for(s.len)) return PK_ERR_INVARIANT;
    for (int32_t b : s.table) {
      if (s.swapped) {
        if (b < 0 || b >= bm->num_host_blocks || host_used[b]) return PK_ERR_INVARIANT;
        host_used[b] = 1;
        ++host_held;
        continue;
      }
      if (b < 0 || b >= bm->num_blocks) return PK_ERR_INVARIANT;
      ++count[b];
    }
  }
  for (int32_t b : bm->host_free) {
    if (b < 0 || b >= bm->num_host_blocks || host_used[b]) return PK_ERR_INVARIANT;
    host_used[b] = 1;
  }
  if (host_held + int64_t(bm->host_free.size()) != bm->num_host_blocks) return PK_ERR_INVARIANT;
  std::vector<char> is_free(bm->num_blocks, 0);
  for (int32_t b : bm->free_stack) {
    if (b < 0 || b >= bm->num_blocks || is_free[b] || count[b] != 0 || bm->entry[b].cached)
      return PK_ERR_INVARIANT;
    is_free[b] = 1;
  }
  int64_t named = 0, cached = 0, idle = 0;
  for (int32_t b = 0; b < bm->num_blocks; ++b) {
    if (count[b] != bm->refs[b]) return PK_ERR_INVARIANT;
    named += count[b] > 0;
    const CacheEntry &e = bm->entry[b];
    if (!e.cached) continue;
    ++cached;
    if (int32_t(e.tokens.size()) != bm->block_size ||
        bm->find_cached(e.chain, e.parent, e.depth, e.tokens.data()) != b)
      return PK_ERR_INVARIANT;
    if (count[b] == 0) {
      if (!bm->idle.count(bm->idle_key(b))) return PK_ERR_INVARIANT;
      ++idle;
    }
  }
  if (cached != int64_t(bm->index.size()) || idle != int64_t(bm->idle.size()))
    return PK_ERR_INVARIANT;
  if (named + int64_t(bm->free_stack.size()) + idle != bm->num_blocks) return PK_ERR_INVARIANT;
  return PK_OK;
}

pk_status pk_bm_stats(const pk_bm *bm, int64_t *live_tokens, int64_t *reserved_slots,
                      int64_t *tail_waste, int32_t *shared_blocks, int64_t *cow_copies) {
  if (!bm) return PK_ERR_INVALID_ARG;
  int64_t live = 0, waste = 0;
  for (const auto &kv : bm->seqs) {
    live += kv.second.len;
    waste += bm->blocks_for(kv.second.len) * bm->block_size - kv.second.len;
  }
  int32_t shared = 0;
  for (int32_t r : bm->refs) shared += r > 1;
  if (live_tokens) *live_tokens = live;
  if (reserved_slots) *reserved_slots = (int64_t(bm->num_blocks) - bm->available()) * bm->block_size;
  if (tail_waste) *tail_waste = waste;
  if (shared_blocks) *shared_blocks = shared;
  if (cow_copies) *cow_copies = bm->cow_copies;
  return PK_OK;
}

pk_status pk_bm_set_swap_space(pk_bm *bm, int32_t num_host_blocks, const int32_t *host_order) {
  if (!bm || num_host_blocks < 0 || bm->num_host_blocks != 0) return PK_ERR_INVALID_ARG;
  try {
    std::vector<int32_t> stack(num_host_blocks);
    std::vector<char> seen(num_host_blocks, 0);
    for (int32_t i = 0; i < num_host_blocks; ++i) {
      const int32_t b = host_order ? host_order[i] : i;
      if (b < 0 || b >= num_host_blocks || seen[b]) return PK_ERR_INVALID_ARG;
      seen[b] = 1;
      stack[num_host_blocks - 1 - i] = b;  // host_order[0] ends on top
    }
    bm->host_free.swap(stack);
  } catch (const std::bad_alloc &) {
    return PK_ERR_NOMEM;
  }
  bm->num_host_blocks = num_host_blocks;
  return PK_OK;
}

pk_status pk_bm_swap_out(pk_bm *bm, int64_t seq_id, int64_t *pairs_out, int32_t cap,
                         int32_t *n_out) {
  if (!bm || !n_out) return PK_ERR_INVALID_ARG;
  *n_out = 0;
  auto it = bm->seqs.find(seq_id);
  if (it == bm->seqs.end()) return PK_ERR_UNKNOWN_SEQ;
  Sequence &s = it->second;
  const int32_t n = int32_t(s.table.size());
  if (s.swapped || cap < n || (n > 0 && !pairs_out)) return PK_ERR_INVALID_ARG;
  if (n > int32_t(bm->host_free.size())) return PK_ERR_OUT_OF_BLOCKS;
  ++bm->clock;
  for (int32_t j = 0; j < n; ++j) {
    const int32_t d = s.table[j];
    const int32_t h = bm->host_free.back();
    bm->host_free.pop_back();
    pairs_out[2 * j] = d;
    pairs_out[2 * j + 1] = h;
    bm->release(d);
    s.table[j] = h;
  }
  s.swapped = true;
  *n_out = n;
  return PK_OK;
}

pk_status pk_bm_swap_in(pk_bm *bm, int64_t seq_id, int64_t *pairs_out, int32_t cap,
                        int32_t *n_out) {
  if (!bm || !n_out) return PK_ERR_INVALID_ARG;
  *n_out = 0;
  auto it = bm->seqs.find(seq_id);
  if (it == bm->seqs.end()) return PK_ERR_UNKNOWN_SEQ;
  Sequence &s = it->second;
  const int32_t n = int32_t(s.table.size());
  if (!s.swapped || cap < n || (n > 0 && !pairs_out)) return PK_ERR_INVALID_ARG;
  if (n > bm->available()) return PK_ERR_OUT_OF_BLOCKS;
  for (int32_t j = 0; j < n; ++j) {
    const int32_t h = s.table[j];
    const int32_t d = bm->take_block();
    bm->refs[d] = 1;
    pairs_out[2 * j] = h;
    pairs_out[2 * j + 1] = d;
    bm->host_free.push_back(h);
    s.table[j] = d;
  }
  s.swapped = false;
  *n_out = n;
  return PK_OK;
}

int32_t pk_bm_is_swapped(const pk_bm *bm, int64_t seq_id) {
  if (!bm) return -1;
  auto it = bm->seqs.find(seq_id);
  return it == bm->seqs.end() ? -1 : (it->second.swapped ? 1 : 0);
}

int32_t pk_bm_host_free(const pk_bm *bm) { return bm ? int32_t(bm->host_free.size()) : -1; }

pk_status pk_bm_cache_match(const pk_bm *bm, const int32_t *tokens, int32_t n,
                            int32_t *n_cached_out) {
  if (!bm || n < 0 || (n > 0 && !tokens) || !n_cached_out) return PK_ERR_INVALID_ARG;
  const int32_t B = bm->block_size;
  uint64_t parent = kChainSeed;
  int32_t j = 0;
  for (; int64_t(j + 1) * B <= n; ++j) {
    const int32_t *tok = tokens + int64_t(j) * B;
    const uint64_t chain = chain_hash(parent, tok, B);
    if (bm->find_cached(chain, parent, j, tok) < 0) break;
    parent = chain;
  }
  *n_cached_out = j * B;
  return PK_OK;
}

pk_status pk_bm_add_seq_cached(pk_bm *bm, int64_t seq_id, const int32_t *tokens, int32_t n,
                               int32_t *n_cached_out) {
  if (!bm || n < 0 || (n > 0 && !tokens)) return PK_ERR_INVALID_ARG;
  if (n_cached_out) *n_cached_out = 0;
  if (bm->seqs.count(seq_id)) return PK_ERR_SEQ_EXISTS;
  const int32_t B = bm->block_size;
  Sequence s;
  try {
    uint64_t parent = kChainSeed;
    for (int32_t j = 0; int64_t(j + 1) * B <= n; ++j) {
      const int32_t *tok = tokens + int64_t(j) * B;
      const uint64_t chain = chain_hash(parent, tok, B);
      const int32_t b = bm->find_cached(chain, parent, j, tok);
      if (b < 0) break;
      s.table.push_back(b);
      parent = chain;
    }
    s.len = int64_t(s.table.size()) * B;
    bm->seqs.emplace(seq_id, s);
  } catch (const std::bad_alloc &) {
    return PK_ERR_NOMEM;
  }
  for (int32_t b : s.table) {
    if (bm->refs[b] == 0) bm->idle.erase(bm->idle_key(b));
    bm->refs[b] += 1;
  }
  bm->cache_hits += int64_t(s.table.size());
  if (n_cached_out) *n_cached_out = int32_t(s.len);
  return PK_OK;
}

pk_status pk_bm_commit(pk_bm *bm, int64_t seq_id, const int32_t *tokens, int32_t n) {
  if (!bm || n < 0 || (n > 0 && !tokens)) return PK_ERR_INVALID_ARG;
  auto it = bm->seqs.find(seq_id);
  if (it == bm->seqs.end()) return PK_ERR_UNKNOWN_SEQ;
  const Sequence &s = it->second;
  if (s.swapped || n > s.len) return PK_ERR_INVALID_ARG;
  const int32_t B = bm->block_size;
  uint64_t parent = kChainSeed;
  try {
    for (int32_t j = 0; int64_t(j + 1) * B <= n; ++j) {
      const int32_t *tok = tokens + int64_t(j) * B;
      const uint64_t chain = chain_hash(parent, tok, B);
      const int32_t b = s.table[j];
      if (!bm->entry[b].cached && bm->find_cached(chain, parent, j, tok) < 0) {
        CacheEntry &e = bm->entry[b];
        e.tokens.assign(tok, tok + B);
        e.depth = j;
        e.chain = chain;
        e.parent = parent;
        bm->index.emplace(chain, b);
        e.cached = true;
      }
      parent = chain;
    }
  } catch (const std::bad_alloc &) {
    return PK_ERR_NOMEM;
  }
  return PK_OK;
}

pk_status pk_bm_cache_stats(const pk_bm *bm, int64_t *cached, int64_t *unreferenced,
                            int64_t *hits, int64_t *evictions) {
  if (!bm) return PK_ERR_INVALID_ARG;
  if (cached) *cached = int64_t(bm->index.size());
  if (unreferenced) *unreferenced = int64_t(bm->idle.size());
  if (hits) *hits = bm->cache_hits;
  if (evictions) *evictions = bm->evictions;
  return PK_OK;
}

pk_status pk_bm_free_blocks(const pk_bm *bm, int32_t *out, int32_t cap, int32_t *n_out) {
  if (!bm || cap < 0 || (cap > 0 && !out) || !n_out) return PK_ERR_INVALID_ARG;
  const int32_t n = int32_t(bm->free_stack.size());
  const int32_t m = std::min(cap, n);
  for (int32_t k = 0; k < m; ++k) out[k] = bm->free_stack[size_t(n - 1 - k)];
  *n_out = n;
  return PK_OK;
}

int32_t pk_bm_is_cached(const pk_bm *bm, int32_t block) {
  if (!bm || block < 0 || block >= bm->num_blocks) return -1;
  return bm->entry[block].cached ? 1 : 0;
}

pk_status pk_bm_prefix_groups(const pk_bm *bm, const int64_t *seq_ids, int32_t n,
                              int32_t max_group_size, int32_t min_prefix_blocks,
                              int32_t *group_offsets, int32_t *group_members,
                              int32_t *group_prefix_len, int32_t *seq_prefix_len,
                              int32_t *num_groups_out) {
  if (!bm || n < 0 || max_group_size < 1 || min_prefix_blocks < 1 || !num_groups_out ||
      (n > 0 && (!seq_ids || !group_offsets || !group_members || !group_prefix_len ||
                 !seq_prefix_len)))
    return PK_ERR_INVALID_ARG;
  *num_groups_out = 0;
  std::vector<const Sequence *> seq(n);
  for (int32_t i = 0; i < n; ++i) {
    auto it = bm->seqs.find(seq_ids[i]);
    if (it == bm->seqs.end()) return PK_ERR_UNKNOWN_SEQ;
    seq[i] = &it->second;
    seq_prefix_len[i] = 0;
  }
  // Sequences whose tables start with the same physical block were forked
  // from one parent; bucket them by that block, keeping batch order.
  std::unordered_map<int32_t, std::vector<int32_t>> buckets;
  std::vector<int32_t> first_seen;
  for (int32_t i = 0; i < n; ++i) {
    if (seq[i]->table.empty() || seq[i]->swapped) continue;
    const int32_t b0 = seq[i]->table[0];
    auto &v = buckets[b0];
    if (v.empty()) first_seen.push_back(b0);
    v.push_back(i);
  }
  const int64_t B = bm->block_size;
  int32_t ng = 0, nm = 0;
  group_offsets[0] = 0;
  for (int32_t b0 : first_seen) {
    const auto &members = buckets[b0];
    for (size_t c0 = 0; c0 < members.size(); c0 += size_t(max_group_size)) {
      const size_t c1 = std::min(members.size(), c0 + size_t(max_group_size));
      if (c1 - c0 < 2) continue;
      // Shared prefix: leading table entries equal across the chunk, limited
      // to blocks every member has filled.
      const Sequence &lead = *seq[members[c0]];
      int64_t common = int64_t(lead.table.size());
      int64_t min_len = lead.len;
      for (size_t k = c0 + 1; k < c1; ++k) {
        const Sequence &o = *seq[members[k]];
        int64_t j = 0;
        const int64_t lim = std::min<int64_t>(common, int64_t(o.table.size()));
        while (j < lim && o.table[j] == lead.table[j]) ++j;
        common = j;
        min_len = std::min(min_len, o.len);
      }
      const int64_t blocks = std::min(common, min_len / B);
      if (blocks < min_prefix_blocks) continue;
      for (size_t k = c0; k < c1; ++k) {
        group_members[nm++] = members[k];
        seq_prefix_len[members[k]] = int32_t(blocks * B);
      }
      group_prefix_len[ng] = int32_t(blocks * B);
      group_offsets[++ng] = nm;
    }
  }
  *num_groups_out = ng;
  return PK_OK;
}

}  // extern "C"
