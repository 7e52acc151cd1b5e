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
#include <stdint.h>

#include <algorithm>
#include <deque>
#include <new>
#include <vector>

#include "pkv.h"

namespace {

struct Request {
  int64_t id;
  int prompt;
  int new_tokens;
  int credits;
};

struct SlotState {
  bool busy = false;
  int64_t id = -1;
  int ctx = 0;          // tokens appended so far
  int decode_left = 0;  // decode steps still to run
  int credits = 0;
};

}  // namespace

struct pkv_sched {
  int num_pages, num_layers, page_tokens, max_context, num_slots, max_blocks;
  std::vector<int32_t> free_list;  // back = next page handed out
  std::deque<Request> queue;
  std::vector<SlotState> slots;
  std::vector<int32_t> block_tables;  // [slot][layer][block]
  int credits_used = 0;
  int assigned = 0;
  pkv_sched_stats stats{};
  // plan buffers (valid until the next step)
  std::vector<int64_t> finished, admitted, append_request;
  std::vector<int32_t> admitted_slot, append_position, append_slot_mapping, decode_slot, context_lens;

  int credits_for(int prompt, int new_tokens) const {
    const int prefix = prompt + new_tokens - 1;
    return ((prefix + page_tokens - 1) / page_tokens) * num_layers;
  }

  int32_t *table(int slot, int layer) { return &block_tables[(size_t(slot) * num_layers + layer) * max_blocks]; }

  // Slot of token `pos` of the request in `slot` at `layer`, taking a page when the
  // token is the first of its block; -1 if the free list is empty.
  int32_t place(int slot, int layer, int pos) {
    int32_t *row = table(slot, layer);
    const int block = pos / page_tokens;
    if (row[block] < 0) {
      if (free_list.empty()) return -1;
      row[block] = free_list.back();
      free_list.pop_back();
      ++assigned;
    }
    return row[block] * page_tokens + pos % page_tokens;
  }

  // Plans the append of token `pos` of slot `slot` in every layer (layer-major
  // slot-mapping buffer is filled in a second pass).
  bool append(int slot, int pos, std::vector<std::vector<int32_t>> &per_layer) {
    for (int l = 0; l < num_layers; ++l) {
      const int32_t m = place(slot, l, pos);
      if (m < 0) return false;
      per_layer[l].push_back(m);
    }
    append_request.push_back(slots[slot].id);
    append_position.push_back(pos);
    return true;
  }

  void retire(int slot) {
    SlotState &st = slots[slot];
    for (int l = 0; l < num_layers; ++l) {
      int32_t *row = table(slot, l);
      for (int b = 0; b < max_blocks; ++b) {
        if (row[b] >= 0) {
          free_list.push_back(row[b]);
          row[b] = -1;
          --assigned;
        }
      }
    }
    credits_used -= st.credits;
    finished.push_back(st.id);
    st = SlotState();
  }
};

extern "C" int pkv_sched_create(int num_pages, int num_layers, int page_tokens, int max_context, int num_slots,
                                const int32_t *free_order, pkv_sched **out) {
  if (out == nullptr) return PKV_ERR_NULL;
  *out = nullptr;
  if (num_pages <= 0 || num_layers <= 0 || page_tokens <= 0 || max_context <= 0 || num_slots <= 0)
    return PKV_ERR_SHAPE;
  pkv_sched *s = new (std::nothrow) pkv_sched();
  if (s == nullptr) return PKV_ERR_SHAPE;
  s->num_pages = num_pages;
  s->num_layers = num_layers;
  s->page_tokens = page_tokens;
  s->max_context = max_context;
  s->num_slots = num_slots;
  s->max_blocks = (max_context + page_tokens - 1) / page_tokens;
  s->free_list.resize(num_pages);
  if (free_order != nullptr) {
    std::vector<char> seen(num_pages, 0);
    for (int i = 0; i < num_pages; ++i) {
      const int32_t p = free_order[i];
      if (p < 0 || p >= num_pages || seen[p]) {
        delete s;
        return PKV_ERR_SHAPE;
      }
      seen[p] = 1;
      s->free_list[i] = p;
    }
  } else {
    for (int i = 0; i < num_pages; ++i) s->free_list[i] = i;
  }
  s->slots.resize(num_slots);
  s->block_tables.assign(size_t(num_slots) * num_layers * s->max_blocks, -1);
  s->context_lens.assign(num_slots, 0);
  s->stats.pool_pages = num_pages;
  s->stats.free_pages = num_pages;
  *out = s;
  return PKV_OK;
}

extern "C" void pkv_sched_destroy(pkv_sched *sched) { delete sched; }

extern "C" int pkv_sched_submit(pkv_sched *s, int64_t request_id, int prompt_tokens, int max_new_tokens) {
  if (s == nullptr) return PKV_ERR_NULL;
  if (prompt_tokens < 1 || prompt_tokens > s->max_context || max_new_tokens < 1) return PKV_ERR_SHAPE;
  const int new_tokens = std::min(max_new_tokens, s->max_context + 1 - prompt_tokens);
  const int credits = s->credits_for(prompt_tokens, new_tokens);
  if (credits > s->num_pages) return PKV_ERR_EXCEEDS_POOL;
  s->queue.push_back(Request{request_id, prompt_tokens, new_tokens, credits});
  s->stats.queued = int32_t(s->queue.size());
  return PKV_OK;
}

extern "C" int pkv_sched_step(pkv_sched *s, pkv_step_plan *plan) {
  if (s == nullptr || plan == nullptr) return PKV_ERR_NULL;
  s->finished.clear();
  s->admitted.clear();
  s->admitted_slot.clear();
  s->append_request.clear();
  s->append_position.clear();
  s->append_slot_mapping.clear();
  s->decode_slot.clear();
  std::fill(s->context_lens.begin(), s->context_lens.end(), 0);
  std::vector<std::vector<int32_t>> per_layer(s->num_layers);

  // (1) retire what finished last step
  for (int i = 0; i < s->num_slots; ++i)
    if (s->slots[i].busy && s->slots[i].decode_left == 0) s->retire(i);

  // (2) admit in FIFO order while a slot is free and the head's credits fit
  bool waited = false;
  while (!s->queue.empty()) {
    int free_slot = -1;
    for (int i = 0; i < s->num_slots; ++i)
      if (!s->slots[i].busy) {
        free_slot = i;
        break;
      }
    if (free_slot < 0) break;
    const Request r = s->queue.front();
    if (s->credits_used + r.credits > s->num_pages) {
      waited = true;
      break;
    }
    s->queue.pop_front();
    SlotState &st = s->slots[free_slot];
    st.busy = true;
    st.id = r.id;
    st.ctx = 0;
    st.decode_left = r.new_tokens - 1;
    st.credits = r.credits;
    s->credits_used += r.credits;
    s->admitted.push_back(r.id);
    s->admitted_slot.push_back(free_slot);
    for (int t = 0; t < r.prompt; ++t)
      if (!s->append(free_slot, t, per_layer)) return PKV_ERR_NO_PAGE;
    st.ctx = r.prompt;
  }
  if (waited) ++s->stats.admission_waits;

  // (3) one decode token per active request with tokens left
  for (int i = 0; i < s->num_slots; ++i) {
    SlotState &st = s->slots[i];
    if (!st.busy || st.decode_left == 0) continue;
    if (!s->append(i, st.ctx, per_layer)) return PKV_ERR_NO_PAGE;
    st.ctx += 1;
    st.decode_left -= 1;
    s->decode_slot.push_back(i);
    s->context_lens[i] = st.ctx;
  }

  for (int l = 0; l < s->num_layers; ++l)
    s->append_slot_mapping.insert(s->append_slot_mapping.end(), per_layer[l].begin(), per_layer[l].end());

  int active = 0;
  for (const SlotState &st : s->slots) active += st.busy;
  pkv_sched_stats &S = s->stats;
  S.peak_active = std::max(S.peak_active, active);
  S.largest_batch = std::max(S.largest_batch, int32_t(s->decode_slot.size()));
  S.peak_pages = std::max(S.peak_pages, s->assigned);
  S.free_pages = int32_t(s->free_list.size());
  S.credits_in_use = s->credits_used;
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
  plan->block_tables = s->block_tables.data();
  plan->max_blocks = s->max_blocks;
  return PKV_OK;
}

extern "C" int pkv_sched_stats_get(const pkv_sched *s, pkv_sched_stats *out) {
  if (s == nullptr || out == nullptr) return PKV_ERR_NULL;
  *out = s->stats;
  return PKV_OK;
}
