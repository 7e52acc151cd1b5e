// Host page allocator and continuous-batching scheduler (C++, no GPU).
//
// Admission policy (samir-vllm README, "Current scope"): a request reserves credits
// for its longest processed prefix, prompt + new - 1 tokens, rounded up to whole
// 16-token pages in every layer, with the new-token budget clamped to the context
// limit; credits are separate from physical pages, which are taken lazily from the
// free list when a block is first written ("tiny-vllm part 3", "Distributing K/V
// into paged blocks": pop from the back, -1 = unassigned).  Requests wait in FIFO
// order while their credits do not fit beside the active ones, so active requests
// always have room to finish; a request larger than the whole pool is rejected.
// On completion a request returns its pages and credits.
//
// pkv_alloc holds the pieces the policy is made of - credits, the free list and the
// block tables - and is exported on its own for callers that schedule themselves;
// pkv_sched adds the FIFO queue, slots and the per-step plan on top of it.
#include <stdint.h>

#include <algorithm>
#include <deque>
#include <new>
#include <vector>

#include "pkv.h"

struct pkv_alloc {
  int num_pages, num_layers, page_tokens, max_context, max_seqs, max_blocks;
  std::vector<int32_t> free_list;     // back = next page handed out
  std::vector<int32_t> block_tables;  // [seq][layer][block], -1 = unassigned
  std::vector<int32_t> seq_credits;   // credits held by each sequence, 0 = not admitted
  std::vector<char> admitted;
  int credits_used = 0;
  int assigned = 0;  // pages currently in some block table

  int credits_for(int prompt, int new_tokens) const {
    const int prefix = prompt + new_tokens - 1;
    return ((prefix + page_tokens - 1) / page_tokens) * num_layers;
  }
  int clamp_new(int prompt, int new_tokens) const { return std::min(new_tokens, max_context + 1 - prompt); }
  int32_t *row(int seq, int layer) { return &block_tables[(size_t(seq) * num_layers + layer) * max_blocks]; }

  // Reserves the credits of a request for `seq`.
  int admit(int seq, int prompt, int new_tokens, int32_t *credits_out) {
    if (seq < 0 || seq >= max_seqs || prompt < 1 || prompt > max_context || new_tokens < 1) return PKV_ERR_SHAPE;
    if (admitted[seq]) return PKV_ERR_STATE;
    const int credits = credits_for(prompt, clamp_new(prompt, new_tokens));
    if (credits_out != nullptr) *credits_out = credits;
    if (credits > num_pages) return PKV_ERR_EXCEEDS_POOL;
    if (credits_used + credits > num_pages) return PKV_ERR_NO_CREDIT;
    admitted[seq] = 1;
    seq_credits[seq] = credits;
    credits_used += credits;
    return PKV_OK;
  }

  // Page of block `block` of (seq, layer), taken from the back of the free list on first use.
  int page(int seq, int layer, int block, int32_t *out) {
    if (seq < 0 || seq >= max_seqs || layer < 0 || layer >= num_layers || block < 0 || block >= max_blocks)
      return PKV_ERR_SHAPE;
    if (!admitted[seq]) return PKV_ERR_STATE;
    int32_t *r = row(seq, layer);
    if (r[block] < 0) {
      if (free_list.empty()) return PKV_ERR_NO_PAGE;
      r[block] = free_list.back();
      free_list.pop_back();
      ++assigned;
    }
    if (out != nullptr) *out = r[block];
    return PKV_OK;
  }

  // Returns the sequence's pages to the free list (layer order, blocks ascending) and its credits.
  int free_seq(int seq) {
    if (seq < 0 || seq >= max_seqs) return PKV_ERR_SHAPE;
    if (!admitted[seq]) return PKV_ERR_STATE;
    for (int l = 0; l < num_layers; ++l) {
      int32_t *r = row(seq, l);
      for (int b = 0; b < max_blocks; ++b) {
        if (r[b] >= 0) {
          free_list.push_back(r[b]);
          r[b] = -1;
          --assigned;
        }
      }
    }
    credits_used -= seq_credits[seq];
    seq_credits[seq] = 0;
    admitted[seq] = 0;
    return PKV_OK;
  }
};

namespace {

// Builds an allocator in *a; PKV_OK or an error (nothing kept on error).
int alloc_init(pkv_alloc *a, int num_pages, int num_layers, int page_tokens, int max_context, int max_seqs,
               const int32_t *free_order) {
  if (num_pages <= 0 || num_layers <= 0 || page_tokens <= 0 || max_context <= 0 || max_seqs <= 0)
    return PKV_ERR_SHAPE;
  a->num_pages = num_pages;
  a->num_layers = num_layers;
  a->page_tokens = page_tokens;
  a->max_context = max_context;
  a->max_seqs = max_seqs;
  a->max_blocks = (max_context + page_tokens - 1) / page_tokens;
  a->free_list.resize(num_pages);
  if (free_order != nullptr) {
    std::vector<char> seen(num_pages, 0);
    for (int i = 0; i < num_pages; ++i) {
      const int32_t p = free_order[i];
      if (p < 0 || p >= num_pages || seen[p]) return PKV_ERR_SHAPE;
      seen[p] = 1;
      a->free_list[i] = p;
    }
  } else {
    for (int i = 0; i < num_pages; ++i) a->free_list[i] = i;
  }
  a->block_tables.assign(size_t(max_seqs) * num_layers * a->max_blocks, -1);
  a->seq_credits.assign(max_seqs, 0);
  a->admitted.assign(max_seqs, 0);
  return PKV_OK;
}

struct Request {
  int64_t id;
  int prompt;
  int new_tokens;
};

struct SlotState {
  bool busy = false;
  int64_t id = -1;
  int ctx = 0;          // tokens appended so far
  int decode_left = 0;  // decode steps still to run
};

}  // namespace

// ---- allocator entry points ---------------------------------------------------------
extern "C" int pkv_alloc_create(int num_pages, int num_layers, int page_tokens, int max_context, int max_seqs,
                                const int32_t *free_order, pkv_alloc **out) {
  if (out == nullptr) return PKV_ERR_NULL;
  *out = nullptr;
  pkv_alloc *a = new (std::nothrow) pkv_alloc();
  if (a == nullptr) return PKV_ERR_SHAPE;
  const int rc = alloc_init(a, num_pages, num_layers, page_tokens, max_context, max_seqs, free_order);
  if (rc != PKV_OK) {
    delete a;
    return rc;
  }
  *out = a;
  return PKV_OK;
}

extern "C" void pkv_alloc_destroy(pkv_alloc *alloc) { delete alloc; }

extern "C" int pkv_alloc_admit(pkv_alloc *alloc, int seq, int prompt_tokens, int max_new_tokens, int32_t *credits) {
  if (alloc == nullptr) return PKV_ERR_NULL;
  return alloc->admit(seq, prompt_tokens, max_new_tokens, credits);
}

extern "C" int pkv_alloc_page(pkv_alloc *alloc, int seq, int layer, int block, int32_t *page) {
  if (alloc == nullptr) return PKV_ERR_NULL;
  return alloc->page(seq, layer, block, page);
}

extern "C" int pkv_alloc_free_seq(pkv_alloc *alloc, int seq) {
  if (alloc == nullptr) return PKV_ERR_NULL;
  return alloc->free_seq(seq);
}

extern "C" const int32_t *pkv_alloc_block_tables(const pkv_alloc *alloc) {
  return alloc == nullptr ? nullptr : alloc->block_tables.data();
}

extern "C" int pkv_alloc_state(const pkv_alloc *alloc, int32_t *free_pages, int32_t *credits_in_use) {
  if (alloc == nullptr) return PKV_ERR_NULL;
  if (free_pages != nullptr) *free_pages = int32_t(alloc->free_list.size());
  if (credits_in_use != nullptr) *credits_in_use = alloc->credits_used;
  return PKV_OK;
}

// ---- scheduler ----------------------------------------------------------------------
struct pkv_sched {
  pkv_alloc alloc;  // slot i of the scheduler is sequence i of the allocator
  std::deque<Request> queue;
  std::vector<SlotState> slots;
  pkv_sched_stats stats{};
  // plan buffers (valid until the next step)
  std::vector<int64_t> finished, admitted, append_request;
  std::vector<int32_t> admitted_slot, append_position, append_slot_mapping, decode_slot, context_lens;

  // Plans the append of token `pos` of slot `slot` in every layer, taking a page when the
  // token is the first of its block (the layer-major slot-mapping buffer is filled in a
  // second pass).
  bool append(int slot, int pos, std::vector<std::vector<int32_t>> &per_layer) {
    const int P = alloc.page_tokens;
    for (int l = 0; l < alloc.num_layers; ++l) {
      int32_t page = -1;
      if (alloc.page(slot, l, pos / P, &page) != PKV_OK) return false;
      per_layer[l].push_back(page * P + pos % P);
    }
    append_request.push_back(slots[slot].id);
    append_position.push_back(pos);
    return true;
  }

  void retire(int slot) {
    alloc.free_seq(slot);
    finished.push_back(slots[slot].id);
    slots[slot] = SlotState();
  }
};

extern "C" int pkv_sched_create(int num_pages, int num_layers, int page_tokens, int max_context, int num_slots,
                                const int32_t *free_order, pkv_sched **out) {
  if (out == nullptr) return PKV_ERR_NULL;
  *out = nullptr;
  pkv_sched *s = new (std::nothrow) pkv_sched();
  if (s == nullptr) return PKV_ERR_SHAPE;
  const int rc = alloc_init(&s->alloc, num_pages, num_layers, page_tokens, max_context, num_slots, free_order);
  if (rc != PKV_OK) {
    delete s;
    return rc;
  }
  s->slots.resize(num_slots);
  s->context_lens.assign(num_slots, 0);
  s->stats.pool_pages = num_pages;
  s->stats.free_pages = num_pages;
  *out = s;
  return PKV_OK;
}

extern "C" void pkv_sched_destroy(pkv_sched *sched) { delete sched; }

extern "C" int pkv_sched_submit(pkv_sched *s, int64_t request_id, int prompt_tokens, int max_new_tokens) {
  if (s == nullptr) return PKV_ERR_NULL;
  const pkv_alloc &a = s->alloc;
  if (prompt_tokens < 1 || prompt_tokens > a.max_context || max_new_tokens < 1) return PKV_ERR_SHAPE;
  const int new_tokens = a.clamp_new(prompt_tokens, max_new_tokens);
  if (a.credits_for(prompt_tokens, new_tokens) > a.num_pages) return PKV_ERR_EXCEEDS_POOL;
  s->queue.push_back(Request{request_id, prompt_tokens, new_tokens});
  s->stats.queued = int32_t(s->queue.size());
  return PKV_OK;
}

extern "C" int pkv_sched_step(pkv_sched *s, pkv_step_plan *plan) {
  if (s == nullptr || plan == nullptr) return PKV_ERR_NULL;
  pkv_alloc &a = s->alloc;
  const int num_slots = a.max_seqs;
  s->finished.clear();
  s->admitted.clear();
  s->admitted_slot.clear();
  s->append_request.clear();
  s->append_position.clear();
  s->append_slot_mapping.clear();
  s->decode_slot.clear();
  std::fill(s->context_lens.begin(), s->context_lens.end(), 0);
  std::vector<std::vector<int32_t>> per_layer(a.num_layers);

  // (1) retire what finished last step
  for (int i = 0; i < num_slots; ++i)
    if (s->slots[i].busy && s->slots[i].decode_left == 0) s->retire(i);

  // (2) admit in FIFO order while a slot is free and the head's credits fit
  bool waited = false;
  while (!s->queue.empty()) {
    int free_slot = -1;
    for (int i = 0; i < num_slots; ++i)
      if (!s->slots[i].busy) {
        free_slot = i;
        break;
      }
    if (free_slot < 0) break;
    const Request r = s->queue.front();
    const int rc = a.admit(free_slot, r.prompt, r.new_tokens, nullptr);
    if (rc == PKV_ERR_NO_CREDIT) {
      waited = true;
      break;
    }
    if (rc != PKV_OK) return PKV_ERR_STATE;
    s->queue.pop_front();
    SlotState &st = s->slots[free_slot];
    st.busy = true;
    st.id = r.id;
    st.ctx = 0;
    st.decode_left = r.new_tokens - 1;
    s->admitted.push_back(r.id);
    s->admitted_slot.push_back(free_slot);
    for (int t = 0; t < r.prompt; ++t)
      if (!s->append(free_slot, t, per_layer)) return PKV_ERR_NO_PAGE;
    st.ctx = r.prompt;
  }
  if (waited) ++s->stats.admission_waits;

  // (3) one decode token per active request with tokens left
  for (int i = 0; i < num_slots; ++i) {
    SlotState &st = s->slots[i];
    if (!st.busy || st.decode_left == 0) continue;
    if (!s->append(i, st.ctx, per_layer)) return PKV_ERR_NO_PAGE;
    st.ctx += 1;
    st.decode_left -= 1;
    s->decode_slot.push_back(i);
    s->context_lens[i] = st.ctx;
  }

  for (int l = 0; l < a.num_layers; ++l)
    s->append_slot_mapping.insert(s->append_slot_mapping.end(), per_layer[l].begin(), per_layer[l].end());

  int active = 0;
  for (const SlotState &st : s->slots) active += st.busy;
  pkv_sched_stats &S = s->stats;
  S.peak_active = std::max(S.peak_active, active);
  S.largest_batch = std::max(S.largest_batch, int32_t(s->decode_slot.size()));
  S.peak_pages = std::max(S.peak_pages, a.assigned);
  S.free_pages = int32_t(a.free_list.size());
  S.credits_in_use = a.credits_used;
  S.active = active;
  S.queued = int32_t(s->queue.size());
  S.steps += 1;

  plan->num_finished = int32_t(s->finished.size());
  plan->finished_request = s->finished.data();
  plan->num_admitted = int32_t(s->admitted.size());
  plan->admitted_request = s->admitted.data();
  plan->admitted_slot = s->admitted_slot.data();
  plan->num_appends = int32_t(s->append_request.size());
  plan->append_request = s->append_request.data();
  plan->append_position = s->append_position.data();
  plan->append_slot_mapping = s->append_slot_mapping.data();
  plan->num_decode = int32_t(s->decode_slot.size());
  plan->decode_slot = s->decode_slot.data();
  plan->context_lens = s->context_lens.data();
  plan->block_tables = a.block_tables.data();
  plan->max_blocks = a.max_blocks;
  return PKV_OK;
}

extern "C" int pkv_sched_stats_get(const pkv_sched *s, pkv_sched_stats *out) {
  if (s == nullptr || out == nullptr) return PKV_ERR_NULL;
  *out = s->stats;
  return PKV_OK;
}
