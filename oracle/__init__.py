"""CPU oracle for paged decode attention (FP64, plain C in ``pkv_oracle.c``).

TEST INFRASTRUCTURE ONLY: the tests, the smoke check and the benchmark's
CPU-baseline leg are the only callers.  The library path never imports this
package.  The oracle shares no code with the CUDA path; its inputs come from the
seeded generators in ``workloads``.

``build()`` compiles the C source with gcc (no fast-math, no FMA contraction, so
x86 and Arm hosts give the same bits); the wrappers below only marshal numpy
arrays into the C entry points.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "pkv_oracle.c")
_LIB = os.path.join(_HERE, "liboracle.so")
_lock = threading.Lock()
_lib = None

ERR_SLOT = 1
ERR_CONTEXT = 2
ERR_PAGE = 4
ERR_ARGS = 8

_P = ctypes.c_void_p
_I = ctypes.c_int
_L = ctypes.c_int64
_D = ctypes.c_double


def build(force: bool = False) -> str:
    """Compile ``liboracle.so`` next to its source (skipped when up to date)."""
    if force or not os.path.exists(_LIB) or os.path.getmtime(_LIB) < os.path.getmtime(_SRC):
        tmp = _LIB + f".tmp{os.getpid()}"
        subprocess.check_call(["gcc", "-std=c99", "-O2", "-ffp-contract=off", "-fno-fast-math",
                               "-shared", "-fPIC", "-o", tmp, _SRC, "-lm"])
        os.replace(tmp, _LIB)
    return _LIB


def _load(path: str):
    L = ctypes.CDLL(path)
    L.oracle_kv_append.argtypes = [_P, _P, _L, _I, _I, _I, _I, _P, _P, _P, _I]
    L.oracle_kv_append.restype = _I
    L.oracle_paged_decode_attention.argtypes = [_P, _P, _L, _I, _I, _I, _I, _P, _I, _P, _L, _P,
                                                _I, _I, _D, _P]
    L.oracle_paged_decode_attention.restype = _I
    L.oracle_attention_weights.argtypes = [_P, _L, _I, _I, _I, _I, _P, _I, _P, _L, _P, _I, _I,
                                           _D, _P]
    L.oracle_attention_weights.restype = _I
    L.oracle_paged_prefill_attention.argtypes = [_P, _P, _L, _I, _I, _I, _I, _P, _I, _P, _P, _L, _P, _I, _I, _D,
                                                 _P]
    L.oracle_paged_prefill_attention.restype = _I
    return L


def use_library(path: str | None):
    """Point the wrappers at another build of the oracle source (mutation tests); None restores."""
    global _lib
    with _lock:
        _lib = _load(path) if path else None


def lib():
    global _lib
    with _lock:
        if _lib is None:
            build()
            _lib = _load(_LIB)
    return _lib


def _ptr(a: np.ndarray):
    assert a.flags["C_CONTIGUOUS"], "oracle inputs must be C-contiguous"
    return a.ctypes.data_as(ctypes.c_void_p)


class Pool:
    """Host copy of a paged pool in the interleaved layout [page][K|V][kv_head][row][dim]."""

    def __init__(self, num_pages: int, page_tokens: int = 16, num_kv_heads: int = 8, head_dim: int = 64,
                 fill: int = 0xFFFF):
        self.num_pages, self.page_tokens = num_pages, page_tokens
        self.num_kv_heads, self.head_dim = num_kv_heads, head_dim
        self.data = np.full((num_pages, 2, num_kv_heads, page_tokens, head_dim), fill, dtype=np.uint16)
        self.page_stride = 2 * num_kv_heads * page_tokens * head_dim

    @property
    def k(self) -> np.ndarray:
        return self.data[:, 0]

    @property
    def v(self) -> np.ndarray:
        return self.data[:, 1]

    def _kv_ptrs(self):
        base = self.data.ctypes.data
        half = self.num_kv_heads * self.page_tokens * self.head_dim * 2
        return ctypes.c_void_p(base), ctypes.c_void_p(base + half)


def kv_append(pool: Pool, k_new: np.ndarray, v_new: np.ndarray, slot_mapping: np.ndarray) -> int:
    k_new = np.ascontiguousarray(k_new, dtype=np.uint16)
    v_new = np.ascontiguousarray(v_new, dtype=np.uint16)
    slots = np.ascontiguousarray(slot_mapping, dtype=np.int32)
    kp, vp = pool._kv_ptrs()
    return lib().oracle_kv_append(kp, vp, pool.page_stride, pool.num_pages, pool.page_tokens,
                                  pool.num_kv_heads, pool.head_dim, _ptr(k_new), _ptr(v_new),
                                  _ptr(slots), int(slots.shape[0]))


def paged_decode_attention(pool: Pool, q: np.ndarray, block_tables: np.ndarray, context_lens: np.ndarray,
                           scale: float, max_context: int, bt_stride: int | None = None):
    """Returns (out float64 [num_seqs, num_q_heads, head_dim], error bits).

    ``block_tables`` is [num_seqs, row] (or any array whose rows are ``bt_stride`` apart).
    """
    q = np.ascontiguousarray(q, dtype=np.uint16)
    bt = np.ascontiguousarray(block_tables, dtype=np.int32)
    lens = np.ascontiguousarray(context_lens, dtype=np.int32)
    num_seqs, num_q_heads, head_dim = q.shape
    if bt_stride is None:
        bt_stride = int(bt.shape[-1]) if bt.ndim > 1 else 0
    out = np.zeros((num_seqs, num_q_heads, head_dim), dtype=np.float64)
    kp, vp = pool._kv_ptrs()
    err = lib().oracle_paged_decode_attention(kp, vp, pool.page_stride, pool.num_pages, pool.page_tokens,
                                              pool.num_kv_heads, head_dim, _ptr(q), num_q_heads, _ptr(bt),
                                              bt_stride, _ptr(lens), num_seqs, max_context, float(scale),
                                              _ptr(out))
    return out, err


def attention_weights(pool: Pool, q: np.ndarray, block_tables: np.ndarray, context_lens: np.ndarray,
                      seq: int, head: int, scale: float, bt_stride: int | None = None):
    q = np.ascontiguousarray(q, dtype=np.uint16)
    bt = np.ascontiguousarray(block_tables, dtype=np.int32)
    lens = np.ascontiguousarray(context_lens, dtype=np.int32)
    num_seqs, num_q_heads, head_dim = q.shape
    if bt_stride is None:
        bt_stride = int(bt.shape[-1])
    w = np.zeros(max(int(lens[seq]), 1), dtype=np.float64)
    kp, _ = pool._kv_ptrs()
    err = lib().oracle_attention_weights(kp, pool.page_stride, pool.num_pages, pool.page_tokens,
                                         pool.num_kv_heads, head_dim, _ptr(q), num_q_heads, _ptr(bt),
                                         bt_stride, _ptr(lens), seq, head, float(scale), _ptr(w))
    return w, err


def paged_prefill_attention(pool: Pool, q: np.ndarray, query_start: np.ndarray, block_tables: np.ndarray,
                            context_lens: np.ndarray, scale: float, max_context: int, bt_stride: int | None = None):
    """Causal attention of the last n_s tokens of each sequence (q rows query_start[s] .. query_start[s+1]-1).

    Returns (out float64 [total, num_q_heads, head_dim], error bits)."""
    q = np.ascontiguousarray(q, dtype=np.uint16)
    qs = np.ascontiguousarray(query_start, dtype=np.int32)
    bt = np.ascontiguousarray(block_tables, dtype=np.int32)
    lens = np.ascontiguousarray(context_lens, dtype=np.int32)
    total, num_q_heads, head_dim = q.shape
    if bt_stride is None:
        bt_stride = int(bt.shape[-1])
    out = np.zeros((total, num_q_heads, head_dim), dtype=np.float64)
    kp, vp = pool._kv_ptrs()
    err = lib().oracle_paged_prefill_attention(kp, vp, pool.page_stride, pool.num_pages, pool.page_tokens,
                                               pool.num_kv_heads, head_dim, _ptr(q), num_q_heads, _ptr(qs), _ptr(bt),
                                               bt_stride, _ptr(lens), int(lens.shape[0]), max_context, float(scale),
                                               _ptr(out))
    return out, err


def decode_workload(wl, layer: int = 0, seqs=None, pool: Pool | None = None):
    """Run the oracle on a ``workloads.configs.DecodeWorkload`` (optionally only on ``seqs``).

    Builds its own pool by appending every token of the chosen sequences, then
    attends.  Returns (out [num_seqs, H, D] float64 with zero rows for sequences
    not chosen, error bits of the attention call, pool).
    """
    if pool is None:
        pool = Pool(wl.num_pages, wl.page_tokens, wl.num_kv_heads, wl.head_dim)
    chosen = range(wl.num_seqs) if seqs is None else seqs
    for s in chosen:
        c = int(wl.context_lens[s])
        if c <= 0 or c > wl.max_blocks * wl.page_tokens:
            continue
        k, v = wl.kv_tokens(s, layer)
        kv_append(pool, k, v, wl.slot_mapping(s, layer, 0, c))
    lens = wl.context_lens.copy()
    if seqs is not None:
        mask = np.zeros(wl.num_seqs, dtype=bool)
        mask[list(seqs)] = True
        lens = np.where(mask, lens, 0).astype(np.int32)
    bt = np.ascontiguousarray(wl.block_tables[:, layer, :])
    out, err = paged_decode_attention(pool, wl.q(layer), bt, lens, wl.scale, wl.max_context)
    return out, err, pool
