// Host BlockManager: free list, reference counts, chained-hash prefix cache,
// LRU evictable pool and atomic allocate/append, as "P06 BlockManager" lays
// them out; fork and copy-on-write as "ans20xx day 31" (`fork_sequence`,
// `ensure_private_last_block`) describes them.
//
// Every operation that can fail checks first and mutates afterwards, so a
// PKV_ERR_OUT_OF_BLOCKS return leaves the manager exactly as it was.
#include <algorithm>
#include <cstdint>
#include <cstring>
#include <deque>
#include <new>
#include <unordered_map>
#include <utility>
#include <vector>

#include "pagedkv.h"

namespace {

constexpr uint64_t kChainStart = 0xFFFFFFFFFFFFFFFFull;  // parent hash of block 0

// FNV-1a over the little-endian bytes of the parent hash and the block's
// tokens, finished with the splitmix64 mixer.  Only equality of hashes is ever
// observed; collisions are not re-verified (the pages do not either).
uint64_t block_hash(uint64_t parent, const int32_t* tokens, int n) {
  uint64_t h = 0xcbf29ce484222325ull;
  auto mix_byte = [&h](uint8_t b) {
    h ^= b;
    h *= 0x100000001b3ull;
  };
  for (int i = 0; i < 8; ++i) mix_byte(static_cast<uint8_t>(parent >> (8 * i)));
  for (int t = 0; t < n; ++t) {
    const uint32_t u = static_cast<uint32_t>(tokens[t]);
    for (int i = 0; i < 4; ++i) mix_byte(static_cast<uint8_t>(u >> (8 * i)));
  }
  h += 0x9e3779b97f4a7c15ull;
  h = (h ^ (h >> 30)) * 0xbf58476d1ce4e5b9ull;
  h = (h ^ (h >> 27)) * 0x94d049bb133111ebull;
  return h ^ (h >> 31);
}

template <class V>
void grow_for_one(V& v) {
  if (v.size() == v.capacity()) v.reserve(v.capacity() < 8 ? 16 : 2 * v.capacity());
}

struct Sequence {
  std::vector<int32_t> table;
  std::vector<int32_t> tokens;
  std::vector<uint64_t> hashes;  // chain over the full blocks
  int64_t cached = 0;            // prefix-cache hits x block_size
};

}  // namespace

struct pkv_block_manager {
  int64_t num_blocks = 0;
  int bs = 16;
  bool prefix = true;

  std::deque<int32_t> free_list;  // unhashed free blocks, FIFO
  std::vector<int32_t> ref;
  std::vector<uint64_t> hash_of;
  std::vector<uint8_t> hashed;  // hash_of[b] is valid
  std::unordered_map<uint64_t, int32_t> hash_to_block;

  // Evictable pool: ref == 0 blocks that keep a hash, as an intrusive doubly
  // linked list in insertion order (head = oldest = next to evict).
  std::vector<int32_t> ev_prev, ev_next;
  std::vector<uint8_t> in_ev;
  int32_t ev_head = -1, ev_tail = -1;
  int64_t ev_count = 0;

  std::unordered_map<int64_t, Sequence> seqs;
  std::vector<std::pair<int64_t, int64_t>> cow_pairs;

  int64_t num_free() const { return static_cast<int64_t>(free_list.size()) + ev_count; }

  void ev_push_back(int32_t b) {
    ev_prev[b] = ev_tail;
    ev_next[b] = -1;
    if (ev_tail >= 0) ev_next[ev_tail] = b; else ev_head = b;
    ev_tail = b;
    in_ev[b] = 1;
    ++ev_count;
  }
  void ev_remove(int32_t b) {
    const int32_t p = ev_prev[b], n = ev_next[b];
    if (p >= 0) ev_next[p] = n; else ev_head = n;
    if (n >= 0) ev_prev[n] = p; else ev_tail = p;
    ev_prev[b] = ev_next[b] = -1;
    in_ev[b] = 0;
    --ev_count;
  }

  // Free list first, else evict the oldest cached block and drop both of its
  // hash records.  Callers have checked capacity.
  int32_t take_block() {
    int32_t b;
    if (!free_list.empty()) {
      b = free_list.front();
      free_list.pop_front();
    } else {
      b = ev_head;
      ev_remove(b);
      auto it = hash_to_block.find(hash_of[b]);
      if (it != hash_to_block.end() && it->second == b) hash_to_block.erase(it);
      hashed[b] = 0;
      hash_of[b] = 0;
    }
    ref[b] = 1;
    return b;
  }

  void register_hash(int32_t b, uint64_t h) {
    hash_of[b] = h;
    hashed[b] = 1;
    hash_to_block.emplace(h, b);  // an existing entry is kept
  }

  void chain(const int32_t* tokens, int64_t n, std::vector<uint64_t>* out) const {
    out->clear();
    uint64_t parent = kChainStart;
    for (int64_t i = 0; i + bs <= n; i += bs) {
      parent = block_hash(parent, tokens + i, bs);
      out->push_back(parent);
    }
  }
};

namespace {
int check_invariants(const pkv_block_manager& bm);
int cow_targets(const int64_t* pairs, int num_pairs, const int32_t* tables, int num_seqs,
                int max_blocks, int32_t* cow_block, int32_t* cow_src);
}  // namespace

extern "C" {

pkv_block_manager* pkv_bm_create(int64_t num_blocks, int block_size, int enable_prefix_cache,
                                 const int32_t* initial_free_order) {
  if (num_blocks < 0 || num_blocks > INT32_MAX || block_size <= 0) return nullptr;
  pkv_block_manager* bm = new (std::nothrow) pkv_block_manager();
  if (!bm) return nullptr;
  try {
    bm->num_blocks = num_blocks;
    bm->bs = block_size;
    bm->prefix = enable_prefix_cache != 0;
    const size_t n = static_cast<size_t>(num_blocks);
    bm->ref.assign(n, 0);
    bm->hash_of.assign(n, 0);
    bm->hashed.assign(n, 0);
    bm->ev_prev.assign(n, -1);
    bm->ev_next.assign(n, -1);
    bm->in_ev.assign(n, 0);
    if (initial_free_order) {
      std::vector<uint8_t> seen(n, 0);
      for (size_t i = 0; i < n; ++i) {
        const int32_t b = initial_free_order[i];
        if (b < 0 || b >= num_blocks || seen[b]) {
          delete bm;
          return nullptr;
        }
        seen[b] = 1;
        bm->free_list.push_back(b);
      }
    } else {
      for (int64_t b = 0; b < num_blocks; ++b) bm->free_list.push_back(static_cast<int32_t>(b));
    }
  } catch (...) {
    delete bm;
    return nullptr;
  }
  return bm;
}

void pkv_bm_destroy(pkv_block_manager* bm) { delete bm; }

int pkv_bm_allocate(pkv_block_manager* bm, int64_t seq_id, const int32_t* tokens,
                    int64_t num_tokens, int32_t* table_out, int64_t table_cap,
                    int64_t* num_table_blocks, int64_t* num_cached_tokens) {
  if (!bm || num_tokens < 0 || (num_tokens > 0 && !tokens)) return PKV_ERR_INVALID_ARG;
  try {
    if (bm->seqs.count(seq_id)) return PKV_ERR_INVALID_ARG;
    const int bs = bm->bs;
    const int64_t n_blocks = (num_tokens + bs - 1) / bs;
    if (table_out && table_cap < n_blocks) return PKV_ERR_INVALID_ARG;
    // (1) chained hashes of the full blocks
    std::vector<uint64_t> hashes;
    if (bm->prefix) bm->chain(tokens, num_tokens, &hashes);
    // (2) consecutive hits within the first (len - 1) / bs blocks
    std::vector<int32_t> hits;
    if (bm->prefix && num_tokens > 0) {
      const int64_t matchable = (num_tokens - 1) / bs;
      for (int64_t i = 0; i < matchable && i < static_cast<int64_t>(hashes.size()); ++i) {
        auto it = bm->hash_to_block.find(hashes[i]);
        if (it == bm->hash_to_block.end()) break;
        hits.push_back(it->second);
      }
    }
    // (3) exact capacity check before any write
    const int64_t new_needed = n_blocks - static_cast<int64_t>(hits.size());
    int64_t revived = 0;
    for (int32_t b : hits) revived += (bm->ref[b] == 0);
    if (new_needed > bm->num_free() - revived) return PKV_ERR_OUT_OF_BLOCKS;

    Sequence seq;
    seq.table.reserve(static_cast<size_t>(n_blocks));
    seq.tokens.assign(tokens, tokens + num_tokens);
    // (4) hits leave the evictable pool and gain a reference
    for (int32_t b : hits) {
      if (bm->ref[b] == 0) bm->ev_remove(b);
      ++bm->ref[b];
      seq.table.push_back(b);
    }
    // (5) the rest are taken fresh
    for (int64_t i = 0; i < new_needed; ++i) seq.table.push_back(bm->take_block());
    // (6) register the full blocks that were not hits
    for (size_t i = hits.size(); i < hashes.size(); ++i) bm->register_hash(seq.table[i], hashes[i]);
    // (7) per-sequence records
    seq.hashes = std::move(hashes);
    seq.cached = static_cast<int64_t>(hits.size()) * bs;
    if (table_out) std::memcpy(table_out, seq.table.data(), sizeof(int32_t) * seq.table.size());
    if (num_table_blocks) *num_table_blocks = static_cast<int64_t>(seq.table.size());
    if (num_cached_tokens) *num_cached_tokens = seq.cached;
    bm->seqs.emplace(seq_id, std::move(seq));
    return PKV_OK;
  } catch (...) {
    return PKV_ERR_INVALID_ARG;
  }
}

int pkv_bm_append_slot(pkv_block_manager* bm, int64_t seq_id, int32_t token, int64_t* slot_out) {
  if (!bm) return PKV_ERR_INVALID_ARG;
  try {
    auto it = bm->seqs.find(seq_id);
    if (it == bm->seqs.end()) return PKV_ERR_BAD_INDEX;
    Sequence& s = it->second;
    const int bs = bm->bs;
    const int64_t pos = static_cast<int64_t>(s.tokens.size());
    const bool boundary = pos / bs == static_cast<int64_t>(s.table.size());
    const bool cow = !boundary && bm->ref[s.table.back()] > 1;
    // (1) a new or private block first: the only step that can fail
    if ((boundary || cow) && bm->num_free() == 0) return PKV_ERR_OUT_OF_BLOCKS;
    // room for one more entry, reserved before anything changes so the
    // push_backs below cannot throw; grown geometrically (reserve(n) allocates
    // exactly n, which would copy the vectors on every append)
    grow_for_one(s.table);
    grow_for_one(s.tokens);
    grow_for_one(s.hashes);
    if (boundary) {
      s.table.push_back(bm->take_block());
    } else if (cow) {
      const int32_t fresh = bm->take_block();
      const int32_t old = s.table.back();
      --bm->ref[old];
      s.table.back() = fresh;
      bm->cow_pairs.emplace_back(old, fresh);
    }
    // (2) then the token
    s.tokens.push_back(token);
    // (3) a block that just filled up joins the chain and the cache
    if (bm->prefix && (pos + 1) % bs == 0) {
      const uint64_t parent = s.hashes.empty() ? kChainStart : s.hashes.back();
      const uint64_t h = block_hash(parent, s.tokens.data() + (pos + 1 - bs), bs);
      s.hashes.push_back(h);
      bm->register_hash(s.table[pos / bs], h);
    }
    if (slot_out) *slot_out = static_cast<int64_t>(s.table[pos / bs]) * bs + pos % bs;
    return PKV_OK;
  } catch (...) {
    return PKV_ERR_INVALID_ARG;
  }
}

int pkv_bm_append_slots(pkv_block_manager* bm, const int64_t* seq_ids, const int32_t* tokens,
                        int64_t n, int64_t* slots_out, int64_t* num_done) {
  if (num_done) *num_done = 0;
  if (!bm || n < 0 || (n > 0 && (!seq_ids || !tokens))) return PKV_ERR_INVALID_ARG;
  for (int64_t i = 0; i < n; ++i) {
    int64_t slot = -1;
    const int rc = pkv_bm_append_slot(bm, seq_ids[i], tokens[i], &slot);
    if (rc != PKV_OK) return rc;
    if (slots_out) slots_out[i] = slot;
    if (num_done) *num_done = i + 1;
  }
  return PKV_OK;
}

int pkv_bm_fork(pkv_block_manager* bm, int64_t parent_id, int64_t child_id) {
  if (!bm) return PKV_ERR_INVALID_ARG;
  try {
    auto it = bm->seqs.find(parent_id);
    if (it == bm->seqs.end()) return PKV_ERR_BAD_INDEX;
    if (bm->seqs.count(child_id)) return PKV_ERR_INVALID_ARG;
    Sequence child = it->second;  // table, tokens, hash chain, cached count
    for (int32_t b : child.table) ++bm->ref[b];
    bm->seqs.emplace(child_id, std::move(child));
    return PKV_OK;
  } catch (...) {
    return PKV_ERR_INVALID_ARG;
  }
}

int pkv_bm_free(pkv_block_manager* bm, int64_t seq_id) {
  if (!bm) return PKV_ERR_INVALID_ARG;
  try {
    auto it = bm->seqs.find(seq_id);
    if (it == bm->seqs.end()) return PKV_OK;
    const std::vector<int32_t>& table = it->second.table;
    for (auto b = table.rbegin(); b != table.rend(); ++b) {
      if (--bm->ref[*b] == 0) {
        if (bm->hashed[*b]) bm->ev_push_back(*b);  // newest end of the LRU pool
        else bm->free_list.push_back(*b);          // (may allocate)
      }
    }
    bm->seqs.erase(it);
    return PKV_OK;
  } catch (...) {  // the free list could not grow: no exception crosses the C ABI
    return PKV_ERR_INVALID_ARG;
  }
}

int pkv_bm_slot(const pkv_block_manager* bm, int64_t seq_id, int64_t pos, int64_t* slot_out) {
  if (!bm || !slot_out) return PKV_ERR_INVALID_ARG;
  auto it = bm->seqs.find(seq_id);
  if (it == bm->seqs.end() || pos < 0) return PKV_ERR_BAD_INDEX;
  const std::vector<int32_t>& table = it->second.table;
  if (pos / bm->bs >= static_cast<int64_t>(table.size())) return PKV_ERR_BAD_INDEX;
  *slot_out = static_cast<int64_t>(table[pos / bm->bs]) * bm->bs + pos % bm->bs;
  return PKV_OK;
}

int64_t pkv_bm_num_free_blocks(const pkv_block_manager* bm) {
  return bm ? bm->num_free() : PKV_ERR_INVALID_ARG;
}

int pkv_bm_can_allocate(const pkv_block_manager* bm, int64_t num_tokens) {
  if (!bm || num_tokens < 0) return 0;
  return (num_tokens + bm->bs - 1) / bm->bs <= bm->num_free() ? 1 : 0;
}

int64_t pkv_bm_block_table(const pkv_block_manager* bm, int64_t seq_id, int32_t* out, int64_t cap) {
  if (!bm) return PKV_ERR_INVALID_ARG;
  auto it = bm->seqs.find(seq_id);
  if (it == bm->seqs.end()) return PKV_ERR_BAD_INDEX;
  const std::vector<int32_t>& t = it->second.table;
  const int64_t n = static_cast<int64_t>(t.size());
  const int64_t k = std::max<int64_t>(0, std::min(n, cap));  // a negative cap copies nothing
  if (out && k > 0) std::memcpy(out, t.data(), sizeof(int32_t) * static_cast<size_t>(k));
  return n;
}

int64_t pkv_bm_num_tokens(const pkv_block_manager* bm, int64_t seq_id) {
  if (!bm) return PKV_ERR_INVALID_ARG;
  auto it = bm->seqs.find(seq_id);
  return it == bm->seqs.end() ? PKV_ERR_BAD_INDEX : static_cast<int64_t>(it->second.tokens.size());
}

int64_t pkv_bm_num_cached_tokens(const pkv_block_manager* bm, int64_t seq_id) {
  if (!bm) return PKV_ERR_INVALID_ARG;
  auto it = bm->seqs.find(seq_id);
  return it == bm->seqs.end() ? PKV_ERR_BAD_INDEX : it->second.cached;
}

int pkv_bm_fill_block_tables(const pkv_block_manager* bm, const int64_t* seq_ids, int64_t n,
                             int32_t* tables_out, int64_t max_blocks, int32_t pad,
                             int32_t* context_lens_out) {
  if (!bm || n < 0 || max_blocks < 0 || (n > 0 && (!seq_ids || !tables_out)))
    return PKV_ERR_INVALID_ARG;
  for (int64_t i = 0; i < n; ++i) {
    auto it = bm->seqs.find(seq_ids[i]);
    if (it == bm->seqs.end()) return PKV_ERR_BAD_INDEX;
    const std::vector<int32_t>& t = it->second.table;
    if (static_cast<int64_t>(t.size()) > max_blocks) return PKV_ERR_INVALID_ARG;
    int32_t* row = tables_out + i * max_blocks;
    std::memcpy(row, t.data(), sizeof(int32_t) * t.size());
    for (int64_t j = static_cast<int64_t>(t.size()); j < max_blocks; ++j) row[j] = pad;
    if (context_lens_out) {
      const size_t len = it->second.tokens.size();
      if (len > static_cast<size_t>(INT32_MAX)) return PKV_ERR_INVALID_ARG;
      context_lens_out[i] = static_cast<int32_t>(len);
    }
  }
  return PKV_OK;
}

int64_t pkv_bm_take_cow_pairs(pkv_block_manager* bm, int64_t* out, int64_t cap_pairs) {
  if (!bm) return PKV_ERR_INVALID_ARG;
  const int64_t n = static_cast<int64_t>(bm->cow_pairs.size());
  if (out && cap_pairs >= n) {
    for (int64_t i = 0; i < n; ++i) {
      out[2 * i] = bm->cow_pairs[i].first;
      out[2 * i + 1] = bm->cow_pairs[i].second;
    }
    bm->cow_pairs.clear();
  }
  return n;
}

int64_t pkv_bm_free_list(const pkv_block_manager* bm, int32_t* out, int64_t cap) {
  if (!bm) return PKV_ERR_INVALID_ARG;
  int64_t i = 0;
  for (int32_t b : bm->free_list) {
    if (out && i < cap) out[i] = b;
    ++i;
  }
  return i;
}

int64_t pkv_bm_evictable_list(const pkv_block_manager* bm, int32_t* out, int64_t cap) {
  if (!bm) return PKV_ERR_INVALID_ARG;
  int64_t i = 0;
  for (int32_t b = bm->ev_head; b >= 0; b = bm->ev_next[b]) {
    if (out && i < cap) out[i] = b;
    ++i;
  }
  return i;
}

int64_t pkv_bm_ref_counts(const pkv_block_manager* bm, int32_t* out, int64_t cap) {
  if (!bm) return PKV_ERR_INVALID_ARG;
  const int64_t n = bm->num_blocks;
  const int64_t k = std::max<int64_t>(0, std::min(n, cap));  // a negative cap copies nothing
  if (out && k > 0) std::memcpy(out, bm->ref.data(), sizeof(int32_t) * static_cast<size_t>(k));
  return n;
}

int pkv_bm_check_invariants(const pkv_block_manager* bm) {
  if (!bm) return PKV_ERR_INVALID_ARG;
  try {
    return check_invariants(*bm);
  } catch (...) {  // scratch arrays could not be allocated
    return PKV_ERR_INVALID_ARG;
  }
}

}  // extern "C"

namespace {
int check_invariants(const pkv_block_manager& bmr) {
  const pkv_block_manager* bm = &bmr;
  const int64_t nb = bm->num_blocks;
  std::vector<uint8_t> in_free(static_cast<size_t>(nb), 0);
  for (int32_t b : bm->free_list) {
    if (in_free[b] || bm->in_ev[b] || bm->ref[b] != 0) return 1;  // I1
    in_free[b] = 1;
  }
  int64_t walked = 0;
  for (int32_t b = bm->ev_head; b >= 0; b = bm->ev_next[b]) {
    if (bm->ref[b] != 0 || !bm->in_ev[b]) return 1;  // I1
    if (++walked > nb) return 1;
  }
  if (walked != bm->ev_count) return 1;
  for (int64_t b = 0; b < nb; ++b)
    if ((bm->in_ev[b] != 0) != (bm->ref[b] == 0 && bm->hashed[b] != 0)) return 2;  // I2
  for (const auto& kv : bm->hash_to_block)
    if (!bm->hashed[kv.second] || bm->hash_of[kv.second] != kv.first) return 3;  // I3
  std::vector<int32_t> count(static_cast<size_t>(nb), 0);
  for (const auto& kv : bm->seqs)
    for (int32_t b : kv.second.table) ++count[b];
  for (int64_t b = 0; b < nb; ++b) {
    if (count[b] != bm->ref[b]) return 4;  // I4
    if (count[b] == 0 && !in_free[b] && !bm->in_ev[b]) return 4;  // leaked block
  }
  if (bm->seqs.empty() && bm->num_free() != nb) return 4;
  for (const auto& kv : bm->seqs) {
    const Sequence& s = kv.second;
    if (s.cached % bm->bs != 0) return 5;  // I5
    if (s.cached > 0 && s.cached >= static_cast<int64_t>(s.tokens.size())) return 5;
  }
  return 0;
}
}  // namespace

// ---- shared-prefix group planning (host) -----------------------------------------
// Consecutive sequences whose tables start with the same physical block form a
// group of at most max_members; the group shares the longest run of leading
// blocks every member has in common with its first member, cut to a multiple
// of lcm(16, block_size) tokens and to the shortest member's context.
extern "C" int pkv_plan_shared_prefix_groups(const int32_t* tables, const int32_t* context_lens,
                                             int num_seqs, int max_blocks, int block_size,
                                             int max_members, int32_t* group_first,
                                             int32_t* seq_group, int32_t* group_shared,
                                             int* num_groups, int* max_shared_tokens,
                                             int* max_own_tokens) {
  if (num_seqs < 0 || max_blocks <= 0 || block_size <= 0 || max_members <= 0 || !num_groups ||
      !max_shared_tokens || !max_own_tokens)
    return PKV_ERR_INVALID_ARG;
  if (num_seqs > 0 && (!tables || !context_lens || !group_first || !seq_group || !group_shared))
    return PKV_ERR_INVALID_ARG;
  int64_t unit = 16;
  while (unit % block_size) unit += 16;  // lcm(16, block_size) for the sizes in use
  int groups = 0, max_shared = 0, max_own = 0;
  int s = 0;
  while (s < num_seqs) {
    const int32_t* lead = tables + static_cast<int64_t>(s) * max_blocks;
    int e = s + 1;
    while (e < num_seqs && e - s < max_members && context_lens[s] > 0 && context_lens[e] > 0 &&
           tables[static_cast<int64_t>(e) * max_blocks] == lead[0])
      ++e;
    int64_t shared = 0;
    if (e - s > 1) {
      int64_t min_len = context_lens[s];
      for (int m = s + 1; m < e; ++m) min_len = std::min<int64_t>(min_len, context_lens[m]);
      int64_t lcp = (min_len + block_size - 1) / block_size;
      lcp = std::min<int64_t>(lcp, max_blocks);
      for (int m = s + 1; m < e; ++m) {
        const int32_t* row = tables + static_cast<int64_t>(m) * max_blocks;
        int64_t k = 0;
        while (k < lcp && row[k] == lead[k]) ++k;
        lcp = k;
      }
      shared = std::min<int64_t>(lcp * block_size, min_len);
      shared -= shared % unit;
    }
    group_first[groups] = s;
    group_shared[groups] = static_cast<int32_t>(shared);
    for (int m = s; m < e; ++m) {
      seq_group[m] = groups;
      max_own = std::max<int>(max_own, static_cast<int>(context_lens[m] - shared));
    }
    max_shared = std::max<int>(max_shared, static_cast<int>(shared));
    ++groups;
    s = e;
  }
  group_first[groups] = num_seqs;
  *num_groups = groups;
  *max_shared_tokens = max_shared;
  *max_own_tokens = max_own;
  return PKV_OK;
}

// ---- copy-on-write targets for the folded copy (host) ------------------------------
// Each pair's dst is a private block (reference count 1 after the copy), so it
// names exactly one (sequence, logical block); the fused _cow launches take
// one such block per sequence.
extern "C" int pkv_cow_targets(const int64_t* pairs, int num_pairs, const int32_t* tables,
                               int num_seqs, int max_blocks, int32_t* cow_block,
                               int32_t* cow_src) {
  if (num_pairs < 0 || num_seqs < 0 || max_blocks <= 0) return PKV_ERR_INVALID_ARG;
  if (num_seqs > 0 && (!tables || !cow_block || !cow_src)) return PKV_ERR_INVALID_ARG;
  if (num_pairs > 0 && !pairs) return PKV_ERR_INVALID_ARG;
  for (int s = 0; s < num_seqs; ++s) cow_block[s] = cow_src[s] = -1;
  try {
    return cow_targets(pairs, num_pairs, tables, num_seqs, max_blocks, cow_block, cow_src);
  } catch (...) {  // the lookup table could not be allocated
    return PKV_ERR_INVALID_ARG;
  }
}

namespace {
int cow_targets(const int64_t* pairs, int num_pairs, const int32_t* tables, int num_seqs,
                int max_blocks, int32_t* cow_block, int32_t* cow_src) {
  struct Target {
    int64_t src;
    int hits;
  };
  std::unordered_map<int64_t, Target> by_dst;
  by_dst.reserve(static_cast<size_t>(num_pairs) * 2);
  for (int i = 0; i < num_pairs; ++i) {
    const int64_t src = pairs[2 * i], dst = pairs[2 * i + 1];
    if (src < 0 || src > INT32_MAX || dst < 0 || dst > INT32_MAX) return PKV_ERR_BAD_INDEX;
    if (!by_dst.emplace(dst, Target{src, 0}).second) return PKV_ERR_BAD_INDEX;
  }
  bool two_in_one = false;
  for (int s = 0; s < num_seqs; ++s) {
    const int32_t* row = tables + static_cast<int64_t>(s) * max_blocks;
    for (int j = 0; j < max_blocks; ++j) {
      if (row[j] < 0) continue;
      const auto it = by_dst.find(row[j]);
      if (it == by_dst.end()) continue;
      ++it->second.hits;
      if (cow_block[s] >= 0) {
        two_in_one = true;
        continue;
      }
      cow_block[s] = j;
      cow_src[s] = static_cast<int32_t>(it->second.src);
    }
  }
  for (const auto& kv : by_dst)
    if (kv.second.hits != 1) return PKV_ERR_BAD_INDEX;  // in no table, or in two places
  return two_in_one ? PKV_ERR_UNSUPPORTED : PKV_OK;
}
}  // namespace
