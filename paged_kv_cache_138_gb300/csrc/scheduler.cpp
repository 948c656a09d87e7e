// Continuous-batching scheduler (host): the per-step bookkeeping of a decode
// server without a model, after "qaqbuyan: vLLM PagedAttention"
// (`ContinuousBatchingScheduler.step`, `_preempt_request`) and the scheduling
// paragraph of "ans20xx day 31".  One call plans one step on a BlockManager and
// hands back everything the device has to do, in order:
//   1. swap-in pairs and prefill slots of the requests admitted this step,
//   2. swap-out pairs of requests preempted this step,
//   3. copy-on-write pairs,
//   4. the decode batch: sequence ids, positions, sampled tokens, slots,
//      block tables and context lengths for attention.
// Only the public pkv_bm_* calls are used.
#include <algorithm>
#include <cstdint>
#include <cstring>
#include <deque>
#include <new>
#include <unordered_map>
#include <vector>

#include <cuda_runtime.h>

#include "pagedkv.h"

namespace {

struct Request {
  int64_t rid = 0;
  std::vector<int32_t> tokens;  // prompt + generated
  int64_t max_new = 0;
  int64_t generated = 0;
  int64_t preemptions = 0;
  bool swapped = false;
  int64_t decoded_step = -1;  // the step that last gave it a decode token
  std::vector<int64_t> host_blocks;  // swap space holding its blocks while swapped out
  bool done() const { return generated >= max_new; }
};

uint64_t mix64(uint64_t z) {
  z += 0x9e3779b97f4a7c15ull;
  z = (z ^ (z >> 30)) * 0xbf58476d1ce4e5b9ull;
  z = (z ^ (z >> 27)) * 0x94d049bb133111ebull;
  return z ^ (z >> 31);
}

}  // namespace

struct pkv_scheduler {
  pkv_block_manager* bm = nullptr;
  int max_batch = 0, max_blocks = 0, block_size = 16;
  bool swap = false;
  uint64_t seed = 0;
  int vocab = 32000;
  std::unordered_map<int64_t, Request> reqs;
  std::deque<int64_t> waiting;
  std::vector<int64_t> running;
  std::deque<int64_t> host_free;
  std::vector<int32_t> table_buf;
  std::vector<int64_t> pending;  // this step's decode candidates (kept to reuse its storage)
  std::vector<int> order;        // batch order by first block (grouped steps)
  std::vector<int32_t> first_block;
  std::vector<int64_t> scratch64;
  std::vector<int32_t> scratch32;
  int64_t step_no = 0;

  // The token request `rid` "samples" at position `pos` (no model).
  int32_t sample(int64_t rid, int64_t pos) const {
    return static_cast<int32_t>(
        mix64(seed ^ mix64(static_cast<uint64_t>(rid) * 0x100000001b3ull + pos)) %
        static_cast<uint64_t>(vocab));
  }

  const std::vector<int32_t>& table_of(int64_t rid) {
    const int64_t n = pkv_bm_block_table(bm, rid, nullptr, 0);
    table_buf.resize(static_cast<size_t>(n > 0 ? n : 0));
    if (n > 0) pkv_bm_block_table(bm, rid, table_buf.data(), n);
    return table_buf;
  }
};

extern "C" {

pkv_scheduler* pkv_sched_create(pkv_block_manager* bm, int max_batch, int max_blocks_per_seq,
                                int block_size, int preemption_swap, int64_t host_blocks,
                                uint64_t seed, int vocab) {
  if (!bm || max_batch <= 0 || max_blocks_per_seq <= 0 || block_size <= 0 || host_blocks < 0 ||
      vocab <= 0)
    return nullptr;
  pkv_scheduler* s = new (std::nothrow) pkv_scheduler();
  if (!s) return nullptr;
  s->bm = bm;
  s->max_batch = max_batch;
  s->max_blocks = max_blocks_per_seq;
  s->block_size = block_size;
  s->swap = preemption_swap != 0;
  s->seed = seed;
  s->vocab = vocab;
  try {
    for (int64_t b = 0; b < host_blocks; ++b) s->host_free.push_back(b);
  } catch (...) {
    delete s;
    return nullptr;
  }
  return s;
}

void pkv_sched_destroy(pkv_scheduler* s) { delete s; }

int pkv_sched_add_request(pkv_scheduler* s, int64_t rid, const int32_t* prompt, int64_t n,
                          int64_t max_new_tokens) {
  if (!s || !prompt || n <= 0 || max_new_tokens < 0) return PKV_ERR_INVALID_ARG;
  try {
    if (s->reqs.count(rid)) return PKV_ERR_INVALID_ARG;
    if ((n + max_new_tokens + s->block_size - 1) / s->block_size > s->max_blocks)
      return PKV_ERR_INVALID_ARG;  // could never fit its table
    Request r;
    r.rid = rid;
    r.tokens.assign(prompt, prompt + n);
    r.max_new = max_new_tokens;
    s->reqs.emplace(rid, std::move(r));
    s->waiting.push_back(rid);
    return PKV_OK;
  } catch (...) {
    return PKV_ERR_INVALID_ARG;
  }
}

int64_t pkv_sched_num_unfinished(const pkv_scheduler* s) {
  return s ? static_cast<int64_t>(s->waiting.size() + s->running.size()) : PKV_ERR_INVALID_ARG;
}

/* Tokens of a request so far (prompt + generated); returns the count, copies
 * up to cap. */
int64_t pkv_sched_request_tokens(const pkv_scheduler* s, int64_t rid, int32_t* out, int64_t cap) {
  if (!s) return PKV_ERR_INVALID_ARG;
  auto it = s->reqs.find(rid);
  if (it == s->reqs.end()) return PKV_ERR_BAD_INDEX;
  const int64_t n = static_cast<int64_t>(it->second.tokens.size());
  const int64_t k = std::max<int64_t>(0, std::min(n, cap));  // a negative cap copies nothing
  if (out && k > 0)
    std::memcpy(out, it->second.tokens.data(), sizeof(int32_t) * static_cast<size_t>(k));
  return n;
}

int pkv_sched_step(pkv_scheduler* s, pkv_sched_step_out* o) {
  if (!s || !o) return PKV_ERR_INVALID_ARG;
  // capacities are checked before anything changes: a step then cannot run out
  const int64_t most_tokens = static_cast<int64_t>(s->max_batch) * s->max_blocks * s->block_size;
  if (!o->batch_rids || !o->positions || !o->tokens || !o->slots || !o->block_tables ||
      !o->context_lens || !o->prefill_rids || !o->prefill_positions || !o->prefill_slots ||
      !o->swap_in_pairs || !o->swap_out_pairs || !o->cow_pairs ||
      o->prefill_cap < most_tokens ||
      o->swap_cap < static_cast<int64_t>(s->max_batch) * s->max_blocks ||
      o->cow_cap < s->max_batch)
    return PKV_ERR_INVALID_ARG;
  o->num_batch = o->num_prefill = o->num_swap_in = o->num_swap_out = o->num_cow = 0;
  o->num_admitted = o->num_finished = o->num_preempted = 0;
  o->cached_tokens = 0;
  const int bs = s->block_size;
  try {
    // 1. release finished requests
    for (size_t i = 0; i < s->running.size();) {
      Request& r = s->reqs[s->running[i]];
      if (r.done()) {
        pkv_bm_free(s->bm, r.rid);
        s->running.erase(s->running.begin() + static_cast<std::ptrdiff_t>(i));
        ++o->num_finished;
      } else {
        ++i;
      }
    }
    // 2. admit first-come first-served while blocks last
    while (!s->waiting.empty() && static_cast<int>(s->running.size()) < s->max_batch) {
      Request& r = s->reqs[s->waiting.front()];
      const int64_t n = static_cast<int64_t>(r.tokens.size());
      int64_t nblk = 0, cached = 0;
      const int rc = pkv_bm_allocate(s->bm, r.rid, r.tokens.data(), n, nullptr, 0, &nblk, &cached);
      if (rc == PKV_ERR_OUT_OF_BLOCKS) break;
      if (rc != PKV_OK) return rc;
      s->waiting.pop_front();
      o->cached_tokens += cached;
      const std::vector<int32_t>& table = s->table_of(r.rid);
      if (r.swapped) {
        // swap-in: blocks past the prefix-cache hits come back from host memory
        for (size_t i = static_cast<size_t>(cached / bs); i < r.host_blocks.size(); ++i) {
          if (o->num_swap_in >= o->swap_cap) return PKV_ERR_INVALID_ARG;
          o->swap_in_pairs[2 * o->num_swap_in] = r.host_blocks[i];
          o->swap_in_pairs[2 * o->num_swap_in + 1] = table[i];
          ++o->num_swap_in;
        }
        for (int64_t b : r.host_blocks) s->host_free.push_back(b);
        r.host_blocks.clear();
        r.swapped = false;
      } else {
        for (int64_t pos = cached; pos < n; ++pos) {
          if (o->num_prefill >= o->prefill_cap) return PKV_ERR_INVALID_ARG;
          o->prefill_rids[o->num_prefill] = r.rid;
          o->prefill_positions[o->num_prefill] = static_cast<int32_t>(pos);
          o->prefill_slots[o->num_prefill] =
              static_cast<int64_t>(table[pos / bs]) * bs + pos % bs;
          ++o->num_prefill;
        }
      }
      s->running.push_back(r.rid);
      ++o->num_admitted;
    }
    // 3. one decode token per running request; on OutOfBlocks the running
    // request with the most generated tokens among those not yet decoded this
    // step is preempted (p1 picks by that count)
    std::vector<int64_t>& pending = s->pending;
    pending.assign(s->running.begin(), s->running.end());
    const int64_t step_no = ++s->step_no;
    size_t i = 0;
    while (i < pending.size()) {
      Request& r = s->reqs[pending[i]];
      const int64_t pos = static_cast<int64_t>(r.tokens.size());
      const int32_t tok = s->sample(r.rid, pos);
      int64_t slot = -1;
      const int rc = pkv_bm_append_slot(s->bm, r.rid, tok, &slot);
      if (rc == PKV_OK) {
        r.tokens.push_back(tok);
        ++r.generated;
        const int b = o->num_batch++;
        o->batch_rids[b] = r.rid;
        o->positions[b] = static_cast<int32_t>(pos);
        o->tokens[b] = tok;
        o->slots[b] = slot;
        r.decoded_step = step_no;
        ++i;
        continue;
      }
      if (rc != PKV_ERR_OUT_OF_BLOCKS) return rc;
      int64_t victim = -1, best = -1;
      for (int64_t rid : s->running) {
        const Request& c = s->reqs[rid];
        if (c.decoded_step == step_no) continue;  // already decoded this step
        if (c.generated > best) {
          best = c.generated;
          victim = rid;
        }
      }
      Request& v = s->reqs[victim];
      if (s->swap) {
        const std::vector<int32_t>& table = s->table_of(victim);
        const size_t used = (v.tokens.size() + bs - 1) / bs;
        if (s->host_free.size() >= used) {
          for (size_t k = 0; k < used; ++k) {
            if (o->num_swap_out >= o->swap_cap) return PKV_ERR_INVALID_ARG;
            const int64_t hb = s->host_free.front();
            s->host_free.pop_front();
            v.host_blocks.push_back(hb);
            o->swap_out_pairs[2 * o->num_swap_out] = table[k];
            o->swap_out_pairs[2 * o->num_swap_out + 1] = hb;
            ++o->num_swap_out;
          }
          v.swapped = true;
        }
      }
      pkv_bm_free(s->bm, victim);
      s->running.erase(std::find(s->running.begin(), s->running.end(), victim));
      ++v.preemptions;
      s->waiting.push_front(victim);
      ++o->num_preempted;
      if (victim == r.rid) {
        ++i;
      } else {
        pending.erase(std::find(pending.begin() + static_cast<std::ptrdiff_t>(i), pending.end(),
                                victim));
      }
    }
    // 4. copy-on-write pairs, then the batch's tables
    const int64_t ncow = pkv_bm_take_cow_pairs(s->bm, nullptr, 0);
    if (ncow > o->cow_cap) return PKV_ERR_INVALID_ARG;
    if (ncow > 0) pkv_bm_take_cow_pairs(s->bm, o->cow_pairs, o->cow_cap);
    o->num_cow = static_cast<int32_t>(ncow);
    o->num_groups = o->max_shared_tokens = o->max_own_tokens = 0;
    const int B = o->num_batch;
    const bool grouping = B > 0 && o->group_limit > 0;
    if (grouping) {
      // order the batch by first physical block so requests sharing a prompt
      // (prefix-cache hits) sit together; the per-row arrays are permuted here
      // and the tables filled in the final order below
      s->order.resize(static_cast<size_t>(B));
      s->first_block.resize(static_cast<size_t>(B));
      for (int b = 0; b < B; ++b) {
        int32_t first = -1;
        pkv_bm_block_table(s->bm, o->batch_rids[b], &first, 1);
        s->first_block[b] = first;
        s->order[b] = b;
      }
      std::stable_sort(s->order.begin(), s->order.end(),
                       [&](int x, int y) { return s->first_block[x] < s->first_block[y]; });
      auto permute = [&](auto* a, auto& tmp) {
        tmp.assign(a, a + B);
        for (int b = 0; b < B; ++b) a[b] = tmp[s->order[b]];
      };
      permute(o->batch_rids, s->scratch64);
      permute(o->slots, s->scratch64);
      permute(o->positions, s->scratch32);
      permute(o->tokens, s->scratch32);
    }
    if (B > 0) {
      const int rc = pkv_bm_fill_block_tables(s->bm, o->batch_rids, B, o->block_tables,
                                              s->max_blocks, -1, o->context_lens);
      if (rc != PKV_OK) return rc;
    }
    if (grouping) {
      const int mb = s->max_blocks;
      if (!o->group_first || !o->seq_group || !o->group_shared) return PKV_ERR_INVALID_ARG;
      int ng = 0, ms = 0, mo = 0;
      const int rc = pkv_plan_shared_prefix_groups(o->block_tables, o->context_lens, B, mb,
                                                   s->block_size, o->group_limit, o->group_first,
                                                   o->seq_group, o->group_shared, &ng, &ms, &mo);
      if (rc != PKV_OK) return rc;
      o->num_groups = ng;
      o->max_shared_tokens = ms;
      o->max_own_tokens = mo;
    }
    return PKV_OK;
  } catch (...) {
    return PKV_ERR_INVALID_ARG;
  }
}


size_t pkv_sched_meta_bytes(const pkv_scheduler* s) {
  if (!s) return 0;
  const size_t B = static_cast<size_t>(s->max_batch);
  // slots (int64), then int32: tables, context lengths, groups (3 B + 1)
  return B * 8 + (B * s->max_blocks + B + 3 * B + 1) * 4 + 64;
}

}  // extern "C"

namespace {

// Where the step's metadata lives in the device staging area: slots (int64,
// unused by the fused launches), then int32 tables | lengths | group_first |
// seq_group | group_shared.
struct Staging {
  int32_t *tables, *lens, *gfirst, *gseq, *gshared;
};

Staging staging_of(const pkv_scheduler* s, void* meta_ptr) {
  uint8_t* meta = static_cast<uint8_t*>(meta_ptr);
  const size_t MB = static_cast<size_t>(s->max_batch);
  Staging g;
  g.tables = reinterpret_cast<int32_t*>(meta + MB * 8);
  g.lens = g.tables + MB * s->max_blocks;
  g.gfirst = g.lens + MB;
  g.gseq = g.gfirst + MB + 1;
  g.gshared = g.gseq + MB;
  return g;
}

bool grouped_step(const pkv_sched_step_out* o) {
  return o->num_groups > 0 && o->max_shared_tokens > 0;
}

// Host -> device copy of a planned step's tables, lengths and groups: one copy
// when out's arrays lie back to back in the staging layout, else one per array.
int copy_metadata(const pkv_scheduler* s, const pkv_sched_step_out* o, const Staging& g,
                  cudaStream_t st) {
  const int B = o->num_batch;
  const int mb = s->max_blocks;
  const size_t MB = static_cast<size_t>(s->max_batch);
  const bool grouped = grouped_step(o);
  const bool packed = o->context_lens == o->block_tables + MB * mb &&
                      o->group_first == o->context_lens + MB &&
                      o->seq_group == o->group_first + MB + 1 && o->group_shared == o->seq_group + MB;
  if (packed) {
    const size_t n = grouped ? MB * mb + MB + 3 * MB + 1 : MB * mb + MB;
    return cudaMemcpyAsync(g.tables, o->block_tables, sizeof(int32_t) * n,
                           cudaMemcpyHostToDevice, st) == cudaSuccess
               ? PKV_OK
               : PKV_ERR_CUDA;
  }
  if (cudaMemcpyAsync(g.tables, o->block_tables, sizeof(int32_t) * B * mb, cudaMemcpyHostToDevice,
                      st) != cudaSuccess ||
      cudaMemcpyAsync(g.lens, o->context_lens, sizeof(int32_t) * B, cudaMemcpyHostToDevice, st) !=
          cudaSuccess)
    return PKV_ERR_CUDA;
  if (grouped &&
      (cudaMemcpyAsync(g.gfirst, o->group_first, sizeof(int32_t) * (o->num_groups + 1),
                       cudaMemcpyHostToDevice, st) != cudaSuccess ||
       cudaMemcpyAsync(g.gseq, o->seq_group, sizeof(int32_t) * B, cudaMemcpyHostToDevice, st) !=
           cudaSuccess ||
       cudaMemcpyAsync(g.gshared, o->group_shared, sizeof(int32_t) * o->num_groups,
                       cudaMemcpyHostToDevice, st) != cudaSuccess))
    return PKV_ERR_CUDA;
  return PKV_OK;
}

}  // namespace

extern "C" {

int pkv_sched_stage_decode(const pkv_scheduler* s, const pkv_sched_step_out* o,
                           const pkv_decode_launch* d, void* stream) {
  if (!s || !o || !d || !d->meta || d->meta_bytes < pkv_sched_meta_bytes(s))
    return PKV_ERR_INVALID_ARG;
  if (o->num_batch == 0) return PKV_OK;
  return copy_metadata(s, o, staging_of(s, d->meta), static_cast<cudaStream_t>(stream));
}

int pkv_sched_launch_decode(const pkv_scheduler* s, const pkv_sched_step_out* o,
                            const pkv_decode_launch* d, void* stream) {
  if (!s || !o || !d || !d->meta || d->meta_bytes < pkv_sched_meta_bytes(s))
    return PKV_ERR_INVALID_ARG;
  const int B = o->num_batch;
  if (B == 0) return PKV_OK;
  const int mb = s->max_blocks;
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  const Staging g = staging_of(s, d->meta);
  // the fused launches recompute each new token's slot from its table row, so
  // the step's slots stay on the host
  if (!d->meta_staged) {
    const int rc = copy_metadata(s, o, g, st);
    if (rc != PKV_OK) return rc;
  }
  if (grouped_step(o))
    return pkv_paged_attention_decode_grouped_fused(
        d->out, d->q, d->k_new, d->v_new, d->k_cache, d->v_cache, g.tables, g.lens, g.gfirst,
        g.gseq, g.gshared, o->num_groups, o->max_shared_tokens, o->max_own_tokens, B,
        d->num_q_heads, d->num_kv_heads, d->head_dim, s->block_size, d->num_blocks, mb, d->scale,
        d->workspace, d->workspace_bytes, d->dev_err, stream);
  return pkv_paged_attention_decode_fused(d->out, d->q, d->k_new, d->v_new, d->k_cache,
                                          d->v_cache, g.tables, g.lens, B, d->num_q_heads,
                                          d->num_kv_heads, d->head_dim, s->block_size,
                                          d->num_blocks, mb, d->scale, d->workspace,
                                          d->workspace_bytes, d->dev_err, stream);
}

}  // extern "C"
