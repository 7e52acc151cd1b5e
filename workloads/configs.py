"""Seeded synthetic workloads for single-token decode over a paged KV cache.

Every input is drawn here from the counter-based generators of ``workloads.rng``;
no step of the method (appending, paging arithmetic inside a kernel, attention)
is computed in this module.  The shapes follow the Llama 3.2 1B decode setup the
pages describe: 32 query heads sharing 8 KV heads (group of 4), head_dim 64,
16-token pages, a 2048-token context limit and a 128 MiB default pool.

A workload is described by:

* ``context_lens[s]`` - tokens of sequence s (the decode token included);
* ``block_tables[s, l, j]`` - physical page of logical block j of sequence s at
  layer l, -1 where unassigned.  Pages come from one shared free list, a seeded
  permutation of the pool that is popped from its back (last in, first out);
* K/V values of logical token t, drawn per (layer, sequence, token) from
  independent streams, so any sequence can be rebuilt alone;
* the query of each (sequence, layer).

``slot_mapping`` (page * page_tokens + row, the append kernel's input format) is
derived from the block table for the tokens being written.
"""
from __future__ import annotations

import math
from dataclasses import dataclass, field

import numpy as np

from . import rng

NUM_Q_HEADS = 32
NUM_KV_HEADS = 8
HEAD_DIM = 64
PAGE_TOKENS = 16
MAX_CONTEXT = 2048
MAX_BLOCKS = MAX_CONTEXT // PAGE_TOKENS
SCALE = 0.125  # 1 / sqrt(64)
TOKEN_ELEMS = NUM_KV_HEADS * HEAD_DIM  # 512 bf16 per token for K (same for V)
PAGE_BYTES = 2 * PAGE_TOKENS * TOKEN_ELEMS * 2  # K + V, 32 KiB


@dataclass
class DecodeWorkload:
    """One batch of decode-attention inputs (configs Tiny, Llama step, Ragged, Bandwidth)."""

    name: str
    seed: int
    num_pages: int
    num_layers: int
    context_lens: np.ndarray            # int32 [num_seqs]
    block_tables: np.ndarray            # int32 [num_seqs, num_layers, max_blocks]
    spike_prob: float = 0.0             # probability that a K element is scaled x8
    max_context: int = MAX_CONTEXT
    page_tokens: int = PAGE_TOKENS
    num_q_heads: int = NUM_Q_HEADS
    num_kv_heads: int = NUM_KV_HEADS
    head_dim: int = HEAD_DIM
    scale: float = SCALE
    keys: dict = field(default_factory=dict)

    def __post_init__(self) -> None:
        for tag in ("k", "v", "q", "spike"):
            self.keys[tag] = rng.stream_key(self.seed, tag)

    # ---- shapes -------------------------------------------------------
    @property
    def num_seqs(self) -> int:
        return int(self.context_lens.shape[0])

    @property
    def max_blocks(self) -> int:
        return int(self.block_tables.shape[2])

    @property
    def token_elems(self) -> int:
        return self.num_kv_heads * self.head_dim

    def has_pages(self, seq: int) -> bool:
        """False for a context length outside [0, max_blocks * page_tokens] (edge-case tests): no pages."""
        c = int(self.context_lens[seq])
        return 0 <= c <= self.max_blocks * self.page_tokens

    def pages_used(self) -> int:
        return int(sum(math.ceil(int(c) / self.page_tokens) for c in self.context_lens)) * self.num_layers

    # ---- values -------------------------------------------------------
    def _token_index(self, layer: int, seq: int, t0: int) -> int:
        return ((layer * self.num_seqs + seq) * self.max_context + t0) * self.token_elems

    def kv_tokens(self, seq: int, layer: int = 0, t0: int = 0, t1: int | None = None):
        """bf16 bits of K and V for tokens [t0, t1) of (seq, layer): [n, num_kv_heads, head_dim]."""
        if t1 is None:
            t1 = int(self.context_lens[seq])
        n = max(t1 - t0, 0)
        base = self._token_index(layer, seq, t0)
        count = n * self.token_elems
        k = rng.normal_bf16(self.keys["k"], base, count, spike_key=self.keys["spike"],
                            spike_prob=self.spike_prob)
        v = rng.normal_bf16(self.keys["v"], base, count)
        shape = (n, self.num_kv_heads, self.head_dim)
        return k.reshape(shape), v.reshape(shape)

    def kv_all(self, layer: int = 0, upto_offset: int = 0):
        """All tokens of every sequence at ``layer``, concatenated in sequence order.

        ``upto_offset`` = 1 leaves out each sequence's last (decode) token.
        Returns (k, v, slot_mapping) ready for a bulk append.
        """
        ks, vs, slots = [], [], []
        for s in range(self.num_seqs):
            n = int(self.context_lens[s]) - upto_offset
            if n <= 0 or not self.has_pages(s):
                continue
            k, v = self.kv_tokens(s, layer, 0, n)
            ks.append(k)
            vs.append(v)
            slots.append(self.slot_mapping(s, layer, 0, n))
        if not ks:
            shape = (0, self.num_kv_heads, self.head_dim)
            return (np.zeros(shape, np.uint16), np.zeros(shape, np.uint16), np.zeros(0, np.int32))
        return np.concatenate(ks), np.concatenate(vs), np.concatenate(slots)

    def decode_tokens(self, layer: int = 0):
        """The decode token (position ctx-1) of every sequence with ctx >= 1."""
        ks, vs, slots = [], [], []
        for s in range(self.num_seqs):
            c = int(self.context_lens[s])
            if c <= 0 or not self.has_pages(s):
                continue
            k, v = self.kv_tokens(s, layer, c - 1, c)
            ks.append(k)
            vs.append(v)
            slots.append(self.slot_mapping(s, layer, c - 1, c))
        return np.concatenate(ks), np.concatenate(vs), np.concatenate(slots)

    def q(self, layer: int = 0) -> np.ndarray:
        """bf16 bits of the queries at ``layer``: [num_seqs, num_q_heads, head_dim]."""
        n = self.num_seqs * self.num_q_heads * self.head_dim
        bits = rng.normal_bf16(self.keys["q"], layer * n, n)
        return bits.reshape(self.num_seqs, self.num_q_heads, self.head_dim)

    def slot_mapping(self, seq: int, layer: int, t0: int, t1: int) -> np.ndarray:
        """Slot (page * page_tokens + row) of tokens [t0, t1) of (seq, layer)."""
        t = np.arange(t0, t1, dtype=np.int64)
        pages = self.block_tables[seq, layer, t // self.page_tokens].astype(np.int64)
        return (pages * self.page_tokens + t % self.page_tokens).astype(np.int32)

    def algorithmic_bytes(self) -> int:
        """Bytes one attention call must read per layer: K+V of valid tokens, q, used table entries, lens."""
        tok = int(np.sum(self.context_lens))
        kv = tok * 2 * self.token_elems * 2
        qb = self.num_seqs * self.num_q_heads * self.head_dim * 2
        tables = 4 * int(sum(math.ceil(int(c) / self.page_tokens) for c in self.context_lens))
        return kv + qb + tables + 4 * self.num_seqs


def _assign_pages(free: list, context_lens: np.ndarray, num_layers: int, max_blocks: int,
                  page_tokens: int = PAGE_TOKENS) -> np.ndarray:
    """Pop pages off the back of ``free`` for every (layer, seq, block) in that order."""
    num_seqs = context_lens.shape[0]
    bt = np.full((num_seqs, num_layers, max_blocks), -1, dtype=np.int32)
    for layer in range(num_layers):
        for s in range(num_seqs):
            c = int(context_lens[s])
            if c < 0 or c > max_blocks * page_tokens:
                continue  # an invalid length (edge-case tests) gets no pages
            for j in range(math.ceil(c / page_tokens)):
                bt[s, layer, j] = free.pop()
    return bt


def tiny(seed: int = 181) -> DecodeWorkload:
    """1 sequence, 1 layer, context 17 (2 pages: 16 + 1 row), pool of 8 pages."""
    lens = np.array([17], dtype=np.int32)
    free = list(rng.permutation(rng.stream_key(seed, "pages"), 8))
    bt = _assign_pages(free, lens, 1, MAX_BLOCKS)
    return DecodeWorkload("tiny", seed, 8, 1, lens, bt)


def llama_step(seed: int = 182) -> DecodeWorkload:
    """16 layers x batch 4, contexts {128, 512, 1024, 2048}, 4096-page (128 MiB) pool, 1 % K spikes x8."""
    lens = np.array([128, 512, 1024, 2048], dtype=np.int32)
    free = list(rng.permutation(rng.stream_key(seed, "pages"), 4096))
    bt = _assign_pages(free, lens, 16, MAX_BLOCKS)
    return DecodeWorkload("llama_step", seed, 4096, 16, lens, bt, spike_prob=0.01)


def ragged(seed: int = 183, num_seqs: int = 64) -> DecodeWorkload:
    """1 layer, contexts uniform in [1, 2048], pool = ceil(1.1 * pages needed), pages shuffled."""
    lens = rng.uniform_int(rng.stream_key(seed, "lens"), 0, num_seqs, 1, MAX_CONTEXT).astype(np.int32)
    need = int(sum(math.ceil(int(c) / PAGE_TOKENS) for c in lens))
    pool = math.ceil(1.1 * need)
    free = list(rng.permutation(rng.stream_key(seed, "pages"), pool))
    bt = _assign_pages(free, lens, 1, MAX_BLOCKS)
    return DecodeWorkload("ragged", seed, pool, 1, lens, bt)


def bandwidth(seed: int = 184, num_seqs: int = 256, context: int = 2048) -> DecodeWorkload:
    """1 layer, batch 256 x context 2048: 32768 pages (1 GiB of bf16 K/V), pages shuffled."""
    lens = np.full(num_seqs, context, dtype=np.int32)
    pool = num_seqs * math.ceil(context / PAGE_TOKENS)
    free = list(rng.permutation(rng.stream_key(seed, "pages"), pool))
    bt = _assign_pages(free, lens, 1, MAX_BLOCKS)
    return DecodeWorkload("bandwidth", seed, pool, 1, lens, bt)


def custom(seed: int, context_lens, num_pages: int | None = None, num_layers: int = 1,
           spike_prob: float = 0.0, max_blocks: int = MAX_BLOCKS, name: str = "custom") -> DecodeWorkload:
    """Any batch of context lengths (0 allowed) with shuffled pages; used by edge-case tests."""
    lens = np.asarray(context_lens, dtype=np.int32)
    need = int(sum(math.ceil(int(c) / PAGE_TOKENS) for c in lens if 0 <= c <= max_blocks * PAGE_TOKENS)) * num_layers
    pool = num_pages if num_pages is not None else max(need, 1)
    free = list(rng.permutation(rng.stream_key(seed, "pages"), pool))
    bt = _assign_pages(free, lens, num_layers, max_blocks)
    return DecodeWorkload(name, seed, pool, num_layers, lens, bt, spike_prob=spike_prob)


# ---------------------------------------------------------------------------
# Continuous-batching trace (requests only; the schedule is host logic of the
# library and of the oracle's reference model, not of this module).
# ---------------------------------------------------------------------------
@dataclass
class TraceWorkload:
    name: str
    seed: int
    num_slots: int
    num_pages: int
    num_steps: int
    prompt_lens: np.ndarray   # int64 [num_requests]
    new_budgets: np.ndarray   # int64 [num_requests], already clamped to the context limit
    free_order: np.ndarray    # int32 [num_pages], initial free list (popped from the back)
    max_context: int = MAX_CONTEXT
    num_layers: int = 1
    keys: dict = field(default_factory=dict)

    def __post_init__(self) -> None:
        for tag in ("k", "v", "q"):
            self.keys[tag] = rng.stream_key(self.seed, "trace-" + tag)

    @property
    def num_requests(self) -> int:
        return int(self.prompt_lens.shape[0])

    def request_kv(self, req: int, t0: int, t1: int):
        """bf16 bits of K and V of tokens [t0, t1) of request ``req``: [n, 8, 64]."""
        n = t1 - t0
        base = (req * self.max_context + t0) * TOKEN_ELEMS
        k = rng.normal_bf16(self.keys["k"], base, n * TOKEN_ELEMS)
        v = rng.normal_bf16(self.keys["v"], base, n * TOKEN_ELEMS)
        return k.reshape(n, NUM_KV_HEADS, HEAD_DIM), v.reshape(n, NUM_KV_HEADS, HEAD_DIM)

    def step_q(self, step: int, slots: np.ndarray) -> np.ndarray:
        """Queries of step ``step`` for the given slots: [len(slots), 32, 64] bf16 bits."""
        per = NUM_Q_HEADS * HEAD_DIM
        out = np.empty((len(slots), NUM_Q_HEADS, HEAD_DIM), dtype=np.uint16)
        for i, s in enumerate(slots):
            out[i] = rng.normal_bf16(self.keys["q"], (step * self.num_slots + int(s)) * per, per).reshape(
                NUM_Q_HEADS, HEAD_DIM)
        return out


def trace(seed: int = 185, num_slots: int = 32, num_pages: int = 4096, num_steps: int = 1000,
          num_requests: int = 400) -> TraceWorkload:
    """32 slots, 1 layer, prompts U[16, 512], new-token budgets U[1, 512], context capped at 2048."""
    p = rng.uniform_int(rng.stream_key(seed, "prompt"), 0, num_requests, 16, 512)
    n = rng.uniform_int(rng.stream_key(seed, "budget"), 0, num_requests, 1, 512)
    n = np.minimum(n, MAX_CONTEXT + 1 - p)
    order = rng.permutation(rng.stream_key(seed, "pages"), num_pages)
    return TraceWorkload("trace", seed, num_slots, num_pages, num_steps, p, n, order)


CONFIGS = {
    "tiny": tiny,
    "llama_step": llama_step,
    "ragged": ragged,
    "bandwidth": bandwidth,
}
