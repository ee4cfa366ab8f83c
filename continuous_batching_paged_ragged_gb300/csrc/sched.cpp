// Host reference scheduler: generates the per-pass ragged batches; never on the timed GPU path.
//
// Follows "Continuous Batching Is Not a Bigger Batch" (deepconcepts.dev), section "What the scheduler
// does on one step": schedule() runs once per pass in two phases.  Phase one walks running requests in
// arrival order; each asks for num_tokens - num_computed_tokens new tokens (one when decoding, the rest
// of the prompt when prefilling) capped by the pass's token budget -- chunked prefill, so there is no
// separate prefill phase.  Blocks for those tokens are allocated on demand; when allocation fails the
// newest running request is popped, its blocks freed, its status set PREEMPTED and num_computed_tokens
// reset to 0, and it is put back at the head of the waiting queue ("newest out first", recompute from
// scratch).  If the popped request is the one being scheduled, phase one stops.  Phase two admits from
// the waiting queue only when the pass preempted nobody, while the budget lasts and while fewer than
// max_num_seqs requests run -- the only place the cap is read ("Saturation and Capacity", section
// "Runtime capacity control": lowering it drains and never evicts; it must be at least 1).
//
// Readings where the pages say nothing: FIFO admission with head-of-line blocking; a pass that computes
// a request's last known token yields one output token; a request with max_output outputs finishes and
// frees its blocks in the same pass; freed blocks join the tail of the free list in block-table order.
//
// Variants (same page, "The allocator is the other half" and "The boundary: when this is worth nothing"):
// RESERVE admits a request only when its whole reservation, ceil((prompt + declared output) / block_size)
// blocks, is free, takes it at admission and returns it at finish, and therefore never preempts;
// UNIT_REQUEST admits only while a batch forms (from a pass that starts with nothing running until the
// first pass in which a member finishes).  A row's block table lists the blocks its context occupies.
//
// Prefix caching (same page, same section: the recompute "is partly refundable" when the freed blocks were
// not evicted): a preempted request's full blocks stay registered while free (returned last block first,
// so its prefix is evicted last); handing a block out evicts it; on readmission the request takes back the
// longest registered prefix, leaving at least one token to compute.
#include <algorithm>
#include <cstdint>
#include <deque>
#include <map>
#include <new>
#include <string>
#include <unordered_map>
#include <vector>

#include "pkv.h"

namespace pkv {
pkv_status fail(pkv_status code, const std::string& msg);
void clear_error();
}  // namespace pkv

namespace {

enum class Status { kWaiting, kRunning, kPreempted, kFinished };

struct Req {
  int64_t id;
  int32_t prompt_len;
  int32_t max_output;
  int32_t declared_output;
  int64_t num_computed = 0;
  int64_t num_output = 0;
  Status status = Status::kWaiting;
  std::vector<int32_t> blocks;
  int64_t num_tokens() const { return (int64_t)prompt_len + num_output; }
};

struct Scheduled {
  Req* req;
  int64_t num_new;
  int64_t start;
};

}  // namespace

struct pkv_sched {
  pkv_sched_config cfg;
  int32_t alloc = PKV_ALLOC_ON_DEMAND;
  int32_t unit = PKV_UNIT_PASS;
  bool batch_open = false;  // UNIT_REQUEST: the current batch still takes members
  bool added_any = false;
  bool prefix_caching = false;
  std::map<std::pair<int64_t, int64_t>, int32_t> cached;  // (request, block j) -> free block still holding it
  std::unordered_map<int32_t, std::pair<int64_t, int64_t>> block_key;  // the reverse map
  std::deque<int32_t> free_list;
  std::vector<Req*> running;       // arrival (admission) order; back = newest
  std::deque<Req*> waiting;        // front = next to admit
  std::unordered_map<int64_t, Req*> live;
  pkv_sched_stats stats{};
  // storage for the last step's arrays
  std::vector<int64_t> req_ids, slot_mapping, preempted, admitted, finished;
  std::vector<int32_t> q_lens, context_lens, qsl, block_tables;

  ~pkv_sched() {
    for (auto& kv : live) delete kv.second;
  }

  int64_t reservation(const Req* r) const {
    return ((int64_t)r->prompt_len + r->declared_output + cfg.block_size - 1) / cfg.block_size;
  }
  // The free list's head; a block handed out no longer holds what it cached.
  int32_t take() {
    const int32_t b = free_list.front();
    free_list.pop_front();
    auto it = block_key.find(b);
    if (it != block_key.end()) {
      cached.erase(it->second);
      block_key.erase(it);
    }
    return b;
  }
  // Blocks at admission: the whole reservation (RESERVE), or the request's cached prefix and those its
  // first new tokens need.  Returns the pass's new tokens, 0 if the request cannot be admitted.
  int64_t admit_blocks(Req* r, int64_t budget) {
    const int64_t bs = cfg.block_size;
    if (alloc == PKV_ALLOC_RESERVE) {
      const int64_t need = reservation(r);
      if (need > (int64_t)free_list.size()) return 0;
      for (int64_t i = 0; i < need; ++i) r->blocks.push_back(take());
      return std::min(r->num_tokens() - r->num_computed, budget);
    }
    std::vector<int32_t> hits;
    while (prefix_caching && r->num_computed == 0) {
      auto it = cached.find({r->id, (int64_t)hits.size()});
      if (it == cached.end() || ((int64_t)hits.size() + 1) * bs > r->num_tokens() - 1) break;
      hits.push_back(it->second);
    }
    const int64_t start = (int64_t)hits.size() * bs;
    const int64_t num_new = std::min(r->num_tokens() - start, budget);
    const int64_t need = (start + num_new + bs - 1) / bs - (int64_t)hits.size();
    if (need > (int64_t)free_list.size() - (int64_t)hits.size()) return 0;
    for (int32_t b : hits) {
      free_list.erase(std::find(free_list.begin(), free_list.end(), b));
      cached.erase(block_key[b]);
      block_key.erase(b);
    }
    r->blocks = hits;
    r->num_computed = start;
    stats.prefix_hit_tokens += start;
    allocate(r, num_new);
    return num_new;
  }

  bool allocate(Req* r, int64_t num_new) {
    const int64_t bs = cfg.block_size;
    const int64_t want = (r->num_computed + num_new + bs - 1) / bs;
    const int64_t need = want - (int64_t)r->blocks.size();
    if (need > (int64_t)free_list.size()) return false;
    for (int64_t i = 0; i < need; ++i) r->blocks.push_back(take());
    return true;
  }

  // Blocks back to the free list's tail; keep registers a preempted request's full blocks for prefix
  // caching and returns them last block first.
  void release(Req* r, bool keep = false) {
    if (keep && prefix_caching) {
      for (size_t j = 0; j < r->blocks.size(); ++j) {
        if ((int64_t)(j + 1) * cfg.block_size <= r->num_computed) {
          cached[{r->id, (int64_t)j}] = r->blocks[j];
          block_key[r->blocks[j]] = {r->id, (int64_t)j};
        }
      }
      for (auto it = r->blocks.rbegin(); it != r->blocks.rend(); ++it) free_list.push_back(*it);
    } else {
      for (int32_t b : r->blocks) free_list.push_back(b);
    }
    r->blocks.clear();
  }
};

using pkv::fail;

extern "C" pkv_status pkv_sched_create(const pkv_sched_config* cfg, const int32_t* free_order, pkv_sched** out) {
  pkv::clear_error();
  if (!cfg || !out) return fail(PKV_ERR_INVALID_ARG, "cfg and out must be non-NULL");
  if (cfg->max_num_seqs < 1) return fail(PKV_ERR_INVALID_ARG, "max_num_seqs must be at least 1");
  if (cfg->token_budget < 1 || cfg->block_size < 1 || cfg->num_blocks < 1)
    return fail(PKV_ERR_INVALID_ARG, "token_budget, block_size and num_blocks must be positive");
  pkv_sched* s = new (std::nothrow) pkv_sched();
  if (!s) return fail(PKV_ERR_INVALID_ARG, "out of host memory");
  s->cfg = *cfg;
  if (free_order) {
    std::vector<char> seen(cfg->num_blocks, 0);
    for (int32_t i = 0; i < cfg->num_blocks; ++i) {
      const int32_t b = free_order[i];
      if (b < 0 || b >= cfg->num_blocks || seen[b]) {
        delete s;
        return fail(PKV_ERR_INVALID_ARG, "free_order must be a permutation of 0..num_blocks-1");
      }
      seen[b] = 1;
      s->free_list.push_back(b);
    }
  } else {
    for (int32_t i = 0; i < cfg->num_blocks; ++i) s->free_list.push_back(i);
  }
  *out = s;
  return PKV_OK;
}

extern "C" void pkv_sched_destroy(pkv_sched* s) { delete s; }

extern "C" pkv_status pkv_sched_add_declared(pkv_sched* s, int64_t req_id, int32_t prompt_len, int32_t max_output,
                                             int32_t declared_output) {
  pkv::clear_error();
  if (!s) return fail(PKV_ERR_INVALID_ARG, "scheduler is NULL");
  if (prompt_len < 1 || max_output < 1) return fail(PKV_ERR_INVALID_ARG, "prompt_len and max_output must be >= 1");
  if (declared_output < max_output) return fail(PKV_ERR_INVALID_ARG, "declared_output must be >= max_output");
  if (s->live.count(req_id)) return fail(PKV_ERR_INVALID_ARG, "duplicate request id");
  const int32_t held = s->alloc == PKV_ALLOC_RESERVE ? declared_output : max_output;
  const int64_t worst = ((int64_t)prompt_len + held + s->cfg.block_size - 1) / s->cfg.block_size;
  if (worst > s->cfg.num_blocks) return fail(PKV_ERR_NO_BLOCKS, "request can never fit the pool");
  Req* r = new Req{req_id, prompt_len, max_output, declared_output};
  s->live[req_id] = r;
  s->waiting.push_back(r);
  s->added_any = true;
  return PKV_OK;
}

extern "C" pkv_status pkv_sched_add(pkv_sched* s, int64_t req_id, int32_t prompt_len, int32_t max_output) {
  return pkv_sched_add_declared(s, req_id, prompt_len, max_output, max_output);
}

extern "C" pkv_status pkv_sched_set_policy(pkv_sched* s, int32_t alloc, int32_t unit) {
  pkv::clear_error();
  if (!s) return fail(PKV_ERR_INVALID_ARG, "scheduler is NULL");
  if (alloc != PKV_ALLOC_ON_DEMAND && alloc != PKV_ALLOC_RESERVE) return fail(PKV_ERR_INVALID_ARG, "unknown alloc");
  if (unit != PKV_UNIT_PASS && unit != PKV_UNIT_REQUEST) return fail(PKV_ERR_INVALID_ARG, "unknown unit");
  if (s->added_any) return fail(PKV_ERR_INVALID_ARG, "set the policy before adding requests");
  if (alloc == PKV_ALLOC_RESERVE && s->prefix_caching)
    return fail(PKV_ERR_INVALID_ARG, "prefix caching refunds recompute; a reserving scheduler never preempts");
  s->alloc = alloc;
  s->unit = unit;
  return PKV_OK;
}

extern "C" pkv_status pkv_sched_set_prefix_caching(pkv_sched* s, int32_t enable) {
  pkv::clear_error();
  if (!s) return fail(PKV_ERR_INVALID_ARG, "scheduler is NULL");
  if (s->added_any) return fail(PKV_ERR_INVALID_ARG, "set prefix caching before adding requests");
  if (enable && s->alloc == PKV_ALLOC_RESERVE)
    return fail(PKV_ERR_INVALID_ARG, "prefix caching refunds recompute; a reserving scheduler never preempts");
  s->prefix_caching = enable != 0;
  return PKV_OK;
}

extern "C" pkv_status pkv_sched_step(pkv_sched* s, pkv_step* out) {
  pkv::clear_error();
  if (!s || !out) return fail(PKV_ERR_INVALID_ARG, "scheduler and out must be non-NULL");
  int64_t budget = s->cfg.token_budget;
  std::vector<Scheduled> sched;
  std::vector<Req*> preempted;
  s->admitted.clear();
  if (s->unit == PKV_UNIT_REQUEST && s->running.empty()) s->batch_open = true;  // a new batch forms

  // phase one: running requests in arrival order
  size_t i = 0;
  while (i < s->running.size() && budget > 0) {
    Req* r = s->running[i];
    const int64_t num_new = std::min(r->num_tokens() - r->num_computed, budget);
    bool schedulable = true;
    while (!s->allocate(r, num_new)) {
      Req* victim = s->running.back();
      s->running.pop_back();
      s->release(victim, /*keep=*/true);
      victim->status = Status::kPreempted;
      s->stats.recomputed_tokens += victim->num_computed;
      s->stats.recomputed_prompt_tokens += std::min<int64_t>(victim->num_computed, victim->prompt_len);
      victim->num_computed = 0;
      s->waiting.push_front(victim);
      preempted.push_back(victim);
      if (victim == r) {
        schedulable = false;
        break;
      }
    }
    if (!schedulable) break;
    sched.push_back({r, num_new, r->num_computed});
    budget -= num_new;
    ++i;
  }

  // phase two: admission, only if this pass preempted nobody (and, per request, while the batch forms)
  if (preempted.empty() && (s->unit == PKV_UNIT_PASS || s->batch_open)) {
    while (!s->waiting.empty() && budget > 0) {
      if ((int64_t)s->running.size() >= s->cfg.max_num_seqs) break;
      Req* r = s->waiting.front();
      const int64_t num_new = s->admit_blocks(r, budget);
      if (num_new == 0) break;  // head-of-line blocking
      s->waiting.pop_front();
      r->status = Status::kRunning;
      s->running.push_back(r);
      s->admitted.push_back(r->id);
      sched.push_back({r, num_new, r->num_computed});
      budget -= num_new;
    }
  }

  // the batch handed to the forward pass
  const int64_t bs = s->cfg.block_size;
  const int32_t B = (int32_t)sched.size();
  int32_t max_blocks = 1;  // a row's table lists the blocks its context occupies (a reservation may hold more)
  for (auto& x : sched) max_blocks = std::max<int32_t>(max_blocks, (int32_t)((x.start + x.num_new + bs - 1) / bs));
  s->req_ids.assign(B, 0);
  s->q_lens.assign(B, 0);
  s->context_lens.assign(B, 0);
  s->qsl.assign(B + 1, 0);
  s->block_tables.assign((size_t)B * max_blocks, -1);
  s->slot_mapping.clear();
  for (int32_t b = 0; b < B; ++b) {
    const Scheduled& x = sched[b];
    s->req_ids[b] = x.req->id;
    s->q_lens[b] = (int32_t)x.num_new;
    s->context_lens[b] = (int32_t)(x.start + x.num_new);
    s->qsl[b + 1] = s->qsl[b] + (int32_t)x.num_new;
    const int64_t used = (x.start + x.num_new + bs - 1) / bs;
    std::copy(x.req->blocks.begin(), x.req->blocks.begin() + used, s->block_tables.begin() + (size_t)b * max_blocks);
    for (int64_t pos = x.start; pos < x.start + x.num_new; ++pos)
      s->slot_mapping.push_back((int64_t)x.req->blocks[pos / bs] * bs + pos % bs);
  }
  s->preempted.clear();
  for (Req* r : preempted) s->preempted.push_back(r->id);

  // the pass has run: advance the scheduled requests
  s->finished.clear();
  for (auto& x : sched) {
    Req* r = x.req;
    r->num_computed += x.num_new;
    if (r->num_computed == r->num_tokens()) {
      r->num_output += 1;
      if (r->num_output >= r->max_output) {
        s->running.erase(std::find(s->running.begin(), s->running.end(), r));
        s->release(r);
        r->status = Status::kFinished;
        s->finished.push_back(r->id);
        s->live.erase(r->id);
        delete r;
      }
    }
  }

  if (!s->finished.empty()) s->batch_open = false;  // a member completed: the batch takes no more
  for (Req* r : s->running) {
    s->stats.live_tokens += r->num_computed;
    s->stats.held_slots += (int64_t)r->blocks.size() * bs;
  }
  s->stats.steps += 1;
  s->stats.preemptions += (int64_t)preempted.size();
  s->stats.max_batch = std::max<int64_t>(s->stats.max_batch, B);
  s->stats.batch_sum += B;
  s->stats.tokens_scheduled += s->qsl[B];

  out->num_seqs = B;
  out->num_tokens = s->qsl[B];
  out->max_blocks_per_seq = max_blocks;
  out->req_ids = s->req_ids.data();
  out->q_lens = s->q_lens.data();
  out->context_lens = s->context_lens.data();
  out->query_start_loc = s->qsl.data();
  out->block_tables = s->block_tables.data();
  out->slot_mapping = s->slot_mapping.data();
  out->num_preempted = (int32_t)s->preempted.size();
  out->preempted = s->preempted.data();
  out->num_admitted = (int32_t)s->admitted.size();
  out->admitted = s->admitted.data();
  out->num_finished = (int32_t)s->finished.size();
  out->finished = s->finished.data();
  return PKV_OK;
}

extern "C" pkv_status pkv_sched_abort(pkv_sched* s, int64_t req_id) {
  pkv::clear_error();
  if (!s) return fail(PKV_ERR_INVALID_ARG, "scheduler is NULL");
  auto it = s->live.find(req_id);
  if (it == s->live.end()) return fail(PKV_ERR_NOT_FOUND, "unknown request id");
  Req* r = it->second;
  auto rit = std::find(s->running.begin(), s->running.end(), r);
  if (rit != s->running.end()) s->running.erase(rit);
  auto wit = std::find(s->waiting.begin(), s->waiting.end(), r);
  if (wit != s->waiting.end()) s->waiting.erase(wit);
  s->release(r);
  s->live.erase(it);
  delete r;
  return PKV_OK;
}

extern "C" pkv_status pkv_sched_set_max_num_seqs(pkv_sched* s, int32_t max_num_seqs) {
  pkv::clear_error();
  if (!s) return fail(PKV_ERR_INVALID_ARG, "scheduler is NULL");
  if (max_num_seqs < 1) return fail(PKV_ERR_INVALID_ARG, "max_num_seqs must be at least 1");
  s->cfg.max_num_seqs = max_num_seqs;
  return PKV_OK;
}

extern "C" void pkv_sched_get_stats(const pkv_sched* s, pkv_sched_stats* out) {
  if (!s || !out) return;
  *out = s->stats;
  out->running = (int32_t)s->running.size();
  out->waiting = (int32_t)s->waiting.size();
  out->free_blocks = (int32_t)s->free_list.size();
}

extern "C" int32_t pkv_sched_done(const pkv_sched* s) {
  return (s && s->running.empty() && s->waiting.empty()) ? 1 : 0;
}

extern "C" int32_t pkv_sched_free_list(const pkv_sched* s, int32_t* out, int32_t n) {
  if (!s) return 0;
  const int32_t cnt = (int32_t)s->free_list.size();
  if (out) {
    for (int32_t i = 0; i < n && i < cnt; ++i) out[i] = s->free_list[i];
  }
  return cnt;
}
