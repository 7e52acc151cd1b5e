"""Reference model of the page-budget admission policy and lazy page assignment.

TEST INFRASTRUCTURE ONLY (like the rest of ``oracle/``): the tests compare the
library's native scheduler with this model step by step.  Written from the pages'
description, plainly, with Python containers:

* samir-vllm README, "Current scope": a request reserves credits for its longest
  processed prefix, prompt + allowed_new - 1 tokens, rounded up to 16-token pages in
  each layer; the allowed output budget is clamped to the context limit; credits are
  separate from the physical pages, which are assigned lazily; requests wait in FIFO
  order when their budget does not fit beside the active ones; a request larger than
  the whole pool is rejected; completion returns both pages and credits.
* tiny-vllm part 3, "Distributing K/V into paged blocks": a page is taken from the
  back of the free list when a block is first written; -1 marks an unassigned block.

Step order (the reading used throughout, stated in the library header too): retire
the requests whose last token was decoded in the previous step (pages pushed back in
layer order, blocks ascending), admit FIFO into the lowest free slots and append each
admitted prompt, then decode one token for every active request with budget left.
A request with budget N decodes N - 1 tokens after its prompt.
"""
from __future__ import annotations

import math
from collections import deque


class Rejected(Exception):
    pass


class AdmissionModel:
    def __init__(self, num_pages, num_layers=1, page_tokens=16, max_context=2048, num_slots=32, free_order=None):
        self.num_pages = num_pages
        self.layers = num_layers
        self.P = page_tokens
        self.max_context = max_context
        self.num_slots = num_slots
        self.max_blocks = math.ceil(max_context / page_tokens)
        self.free = list(range(num_pages)) if free_order is None else [int(p) for p in free_order]
        self.queue = deque()
        self.slot = [None] * num_slots          # None or dict(id, ctx, left, credits)
        self.tables = [[[-1] * self.max_blocks for _ in range(num_layers)] for _ in range(num_slots)]
        self.credits_used = 0
        self.stats = dict(peak_active=0, largest_batch=0, peak_pages=0, admission_waits=0)

    def submit(self, rid, prompt, new):
        if prompt < 1 or prompt > self.max_context or new < 1:
            raise ValueError("bad request")
        new = min(new, self.max_context - prompt + 1)          # clamp to the context limit
        credits = math.ceil((prompt + new - 1) / self.P) * self.layers
        if credits > self.num_pages:
            raise Rejected(rid)
        self.queue.append(dict(id=rid, prompt=prompt, new=new, credits=credits))

    def _write_token(self, s, pos, mapping):
        """Record token `pos` of slot s in every layer, assigning pages lazily."""
        blk, row = divmod(pos, self.P)
        for layer in range(self.layers):
            table = self.tables[s][layer]
            if table[blk] == -1:
                table[blk] = self.free.pop()                      # LIFO
            mapping[layer].append(table[blk] * self.P + row)

    def step(self):
        finished, admitted, admitted_slot = [], [], []
        app_req, app_pos = [], []
        mapping = [[] for _ in range(self.layers)]
        for s in range(self.num_slots):                           # retire
            st = self.slot[s]
            if st is not None and st["left"] == 0:
                for layer in range(self.layers):
                    for b in range(self.max_blocks):
                        if self.tables[s][layer][b] != -1:
                            self.free.append(self.tables[s][layer][b])
                            self.tables[s][layer][b] = -1
                self.credits_used -= st["credits"]
                finished.append(st["id"])
                self.slot[s] = None
        while self.queue:                                          # admit, FIFO
            free_slots = [s for s in range(self.num_slots) if self.slot[s] is None]
            if not free_slots:
                break
            head = self.queue[0]
            if self.credits_used + head["credits"] > self.num_pages:
                self.stats["admission_waits"] += 1
                break
            self.queue.popleft()
            s = free_slots[0]
            self.slot[s] = dict(id=head["id"], ctx=head["prompt"], left=head["new"] - 1, credits=head["credits"])
            self.credits_used += head["credits"]
            admitted.append(head["id"])
            admitted_slot.append(s)
            for pos in range(head["prompt"]):
                self._write_token(s, pos, mapping)
                app_req.append(head["id"])
                app_pos.append(pos)
        decode, lens = [], [0] * self.num_slots
        for s in range(self.num_slots):                           # decode one token each
            st = self.slot[s]
            if st is None or st["left"] == 0:
                continue
            self._write_token(s, st["ctx"], mapping)
            app_req.append(st["id"])
            app_pos.append(st["ctx"])
            st["ctx"] += 1
            st["left"] -= 1
            decode.append(s)
            lens[s] = st["ctx"]
        active = sum(st is not None for st in self.slot)
        self.stats["peak_active"] = max(self.stats["peak_active"], active)
        self.stats["largest_batch"] = max(self.stats["largest_batch"], len(decode))
        self.stats["peak_pages"] = max(self.stats["peak_pages"], self.num_pages - len(self.free))
        return dict(finished=finished, admitted=admitted, admitted_slot=admitted_slot, append_request=app_req,
                    append_position=app_pos, append_slot_mapping=mapping, decode_slot=decode, context_lens=lens,
                    block_tables=[[list(t) for t in per_slot] for per_slot in self.tables])
