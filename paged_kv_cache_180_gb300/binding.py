"""Thin Python binding of the C ABI in ``include/pkv.h`` (argument marshalling only).

Every step of the decode path runs in the CUDA kernels of ``libpkv.so``; this
module only turns tensors into pointers and sizes, passes the current CUDA
stream, and raises on a negative status.  There is no CPU fallback: if the
library is missing the import fails.

Function names follow the C entry points without their ``pkv_`` prefix.
PyTorch provides device memory and streams.
"""
from __future__ import annotations

import ctypes
import os

import torch

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "libpkv.so")

if not os.path.exists(LIB_PATH):
    raise ImportError(f"{LIB_PATH} is missing: build it with `python -m paged_kv_cache_180_gb300.build` "
                      "(the CUDA path has no fallback)")

_lib = ctypes.CDLL(LIB_PATH)

PKV_OK = 0
DEV_BAD_SLOT = 1
DEV_BAD_CONTEXT = 2
DEV_BAD_PAGE = 4
DEV_TIMEOUT = 8


class PkvPool(ctypes.Structure):
    """Mirror of ``pkv_pool``."""
    _fields_ = [("k_base", ctypes.c_void_p), ("v_base", ctypes.c_void_p), ("page_stride_bytes", ctypes.c_int64),
                ("num_pages", ctypes.c_int32), ("page_tokens", ctypes.c_int32),
                ("num_kv_heads", ctypes.c_int32), ("head_dim", ctypes.c_int32)]


class PkvStepPlan(ctypes.Structure):
    """Mirror of ``pkv_step_plan``."""
    _fields_ = [("num_finished", ctypes.c_int32), ("finished_request", ctypes.POINTER(ctypes.c_int64)),
                ("num_admitted", ctypes.c_int32), ("admitted_request", ctypes.POINTER(ctypes.c_int64)),
                ("admitted_slot", ctypes.POINTER(ctypes.c_int32)),
                ("num_appends", ctypes.c_int32), ("append_request", ctypes.POINTER(ctypes.c_int64)),
                ("append_position", ctypes.POINTER(ctypes.c_int32)),
                ("append_slot_mapping", ctypes.POINTER(ctypes.c_int32)),
                ("num_decode", ctypes.c_int32), ("decode_slot", ctypes.POINTER(ctypes.c_int32)),
                ("context_lens", ctypes.POINTER(ctypes.c_int32)), ("block_tables", ctypes.POINTER(ctypes.c_int32)),
                ("max_blocks", ctypes.c_int32)]


class PkvSchedStats(ctypes.Structure):
    """Mirror of ``pkv_sched_stats``."""
    _fields_ = [("pool_pages", ctypes.c_int32), ("peak_active", ctypes.c_int32), ("largest_batch", ctypes.c_int32),
                ("peak_pages", ctypes.c_int32), ("admission_waits", ctypes.c_int32), ("free_pages", ctypes.c_int32),
                ("credits_in_use", ctypes.c_int32), ("active", ctypes.c_int32), ("queued", ctypes.c_int32),
                ("steps", ctypes.c_int64)]


_P, _I, _L, _F, _Z = ctypes.c_void_p, ctypes.c_int, ctypes.c_int64, ctypes.c_float, ctypes.c_size_t
_PP = ctypes.POINTER(PkvPool)

EXPORTS = {
    # name: (restype, argtypes)
    "pkv_kv_pool_bytes": (_Z, [_I, _I, _I, _I]),
    "pkv_kv_pool_create": (_I, [_P, _P, _L, _I, _I, _I, _I, _PP]),
    "pkv_kv_append": (_I, [_PP, _P, _P, _P, _I, _P, _P]),
    "pkv_decode_workspace_bytes": (_Z, [_I, _I, _I]),
    "pkv_paged_decode_attention": (_I, [_PP, _P, _P, _I, _P, _L, _P, _I, _I, _F, _P, _Z, _P, _P]),
    "pkv_paged_decode_attention_ctas": (_I, [_PP, _P, _P, _I, _P, _L, _P, _I, _I, _F, _P, _Z, _P, _I, _P]),
    "pkv_decode_max_ctas": (_I, []),
    "pkv_decode_plan": (_I, [_I, _I, ctypes.POINTER(_I), ctypes.POINTER(_I)]),
    "pkv_status_string": (ctypes.c_char_p, [_I]),
    "pkv_paged_decode_attention_noalloc": (_I, [_PP, _P, _P, _I, _P, _L, _P, _I, _I, _F, _P, _P]),
    "pkv_decode_step": (_I, [_PP, _P, _P, _P, _P, _P, _I, _P, _L, _P, _I, _I, _F, _P, _Z, _P, _P]),
    "pkv_decode_step_ex": (_I, [_PP, _P, _P, _P, _P, _P, _I, _P, _L, _P, _I, _I, _F, _P, _Z, _P, ctypes.c_uint, _P]),
    "pkv_paged_prefill_attention": (_I, [_PP, _P, _P, _I, _I, _P, _P, _L, _P, _I, _I, _I, _F, _P, _P]),
    "pkv_paged_prefill_attention_ex": (_I, [_PP, _P, _P, _I, _I, _P, _P, _L, _P, _I, _I, _I, _F, _P, ctypes.c_uint,
                                            _P]),
    "pkv_alloc_create": (_I, [_I, _I, _I, _I, _I, _P, ctypes.POINTER(_P)]),
    "pkv_alloc_destroy": (None, [_P]),
    "pkv_alloc_admit": (_I, [_P, _I, _I, _I, ctypes.POINTER(ctypes.c_int32)]),
    "pkv_alloc_page": (_I, [_P, _I, _I, _I, ctypes.POINTER(ctypes.c_int32)]),
    "pkv_alloc_free_seq": (_I, [_P, _I]),
    "pkv_alloc_block_tables": (ctypes.POINTER(ctypes.c_int32), [_P]),
    "pkv_alloc_state": (_I, [_P, ctypes.POINTER(ctypes.c_int32), ctypes.POINTER(ctypes.c_int32)]),
    "pkv_sched_create": (_I, [_I, _I, _I, _I, _I, _P, ctypes.POINTER(_P)]),
    "pkv_sched_destroy": (None, [_P]),
    "pkv_sched_submit": (_I, [_P, _L, _I, _I]),
    "pkv_sched_step": (_I, [_P, ctypes.POINTER(PkvStepPlan)]),
    "pkv_sched_stats_get": (_I, [_P, ctypes.POINTER(PkvSchedStats)]),
}

NOALLOC_MAX_SEQS = 512  # PKV_NOALLOC_MAX_SEQS
OVERLAP_PREVIOUS = 1  # PKV_OVERLAP_PREVIOUS

for _name, (_res, _args) in EXPORTS.items():
    _fn = getattr(_lib, _name)
    _fn.restype = _res
    _fn.argtypes = _args


class PkvError(RuntimeError):
    def __init__(self, where: str, code: int):
        super().__init__(f"{where}: {status_string(code)} ({code})")
        self.code = code


def _check(where: str, rc: int) -> None:
    if rc != PKV_OK:
        raise PkvError(where, rc)


def status_string(code: int) -> str:
    return _lib.pkv_status_string(int(code)).decode()


def _stream(stream) -> int:
    if stream is None:
        stream = torch.cuda.current_stream()
    return int(stream.cuda_stream)


def _ptr(t: torch.Tensor | None) -> int | None:
    return None if t is None else int(t.data_ptr())


# ---------------------------------------------------------------------------
def kv_pool_bytes(num_pages: int, page_tokens: int = 16, num_kv_heads: int = 8, head_dim: int = 64) -> int:
    return int(_lib.pkv_kv_pool_bytes(num_pages, page_tokens, num_kv_heads, head_dim))


def kv_pool_create(k_pool: torch.Tensor | int, v_pool: torch.Tensor | int, page_stride_bytes: int, num_pages: int,
                   page_tokens: int = 16, num_kv_heads: int = 8, head_dim: int = 64) -> PkvPool:
    """Descriptor for caller-owned pool memory (tensors or raw device addresses)."""
    kp = k_pool if isinstance(k_pool, int) else _ptr(k_pool)
    vp = v_pool if isinstance(v_pool, int) else _ptr(v_pool)
    desc = PkvPool()
    _check("pkv_kv_pool_create", _lib.pkv_kv_pool_create(kp, vp, page_stride_bytes, num_pages, page_tokens,
                                                         num_kv_heads, head_dim, ctypes.byref(desc)))
    return desc


class KVPool:
    """One interleaved pool buffer ([page][K|V][kv_head][row][dim] bf16) owned by a torch tensor."""

    def __init__(self, num_pages: int, page_tokens: int = 16, num_kv_heads: int = 8, head_dim: int = 64,
                 device="cuda", buffer: torch.Tensor | None = None):
        nbytes = kv_pool_bytes(num_pages, page_tokens, num_kv_heads, head_dim)
        if buffer is None:
            buffer = torch.empty(nbytes // 2, dtype=torch.bfloat16, device=device)
        assert buffer.numel() * buffer.element_size() >= nbytes
        self.buffer = buffer
        self.num_pages, self.page_tokens = num_pages, page_tokens
        self.num_kv_heads, self.head_dim = num_kv_heads, head_dim
        half = num_kv_heads * page_tokens * head_dim * 2
        base = _ptr(buffer)
        self.desc = kv_pool_create(base, base + half, 2 * half, num_pages, page_tokens, num_kv_heads, head_dim)

    def view(self) -> torch.Tensor:
        """The pool as [num_pages, 2, num_kv_heads, page_tokens, head_dim] bf16."""
        return self.buffer[: self.num_pages * 2 * self.num_kv_heads * self.page_tokens * self.head_dim].view(
            self.num_pages, 2, self.num_kv_heads, self.page_tokens, self.head_dim)


def kv_append(pool: KVPool | PkvPool, k_new: torch.Tensor, v_new: torch.Tensor, slot_mapping: torch.Tensor,
              status: torch.Tensor | None = None, stream=None) -> None:
    desc = pool.desc if isinstance(pool, KVPool) else pool
    n = int(slot_mapping.shape[0])
    _check("pkv_kv_append", _lib.pkv_kv_append(ctypes.byref(desc), _ptr(k_new), _ptr(v_new), _ptr(slot_mapping),
                                               n, _ptr(status), _stream(stream)))


def decode_workspace_bytes(num_seqs: int, num_q_heads: int = 32, head_dim: int = 64) -> int:
    return int(_lib.pkv_decode_workspace_bytes(num_seqs, num_q_heads, head_dim))


def decode_workspace(num_seqs: int, device="cuda") -> torch.Tensor:
    """A zero-filled workspace for pkv_paged_decode_attention (zeroed once; calls keep it valid)."""
    return torch.zeros(decode_workspace_bytes(num_seqs), dtype=torch.uint8, device=device)


def decode_max_ctas() -> int:
    return int(_lib.pkv_decode_max_ctas())


def decode_plan(num_seqs: int, max_context: int) -> tuple[int, int]:
    g, n = _I(0), _I(0)
    _check("pkv_decode_plan", _lib.pkv_decode_plan(num_seqs, max_context, ctypes.byref(g), ctypes.byref(n)))
    return g.value, n.value


def paged_decode_attention(pool: KVPool | PkvPool, out: torch.Tensor, q: torch.Tensor, block_tables: torch.Tensor,
                           block_table_stride: int, context_lens: torch.Tensor, max_context: int, scale: float,
                           workspace: torch.Tensor, status: torch.Tensor | None = None, num_ctas: int = 0,
                           stream=None) -> None:
    """out[s, h, :] = softmax(scale * q[s, h] . K[h // group]) V over the cached tokens of sequence s."""
    desc = pool.desc if isinstance(pool, KVPool) else pool
    num_seqs, num_q_heads = int(q.shape[0]), int(q.shape[1])
    ws_bytes = workspace.numel() * workspace.element_size()
    if num_ctas:
        rc = _lib.pkv_paged_decode_attention_ctas(ctypes.byref(desc), _ptr(out), _ptr(q), num_q_heads,
                                                  _ptr(block_tables), block_table_stride, _ptr(context_lens),
                                                  num_seqs, max_context, scale, _ptr(workspace), ws_bytes,
                                                  _ptr(status), num_ctas, _stream(stream))
    else:
        rc = _lib.pkv_paged_decode_attention(ctypes.byref(desc), _ptr(out), _ptr(q), num_q_heads,
                                             _ptr(block_tables), block_table_stride, _ptr(context_lens),
                                             num_seqs, max_context, scale, _ptr(workspace), ws_bytes,
                                             _ptr(status), _stream(stream))
    _check("pkv_paged_decode_attention", rc)


def decode_step(pool: KVPool | PkvPool, k_new: torch.Tensor, v_new: torch.Tensor, slot_mapping: torch.Tensor,
                out: torch.Tensor, q: torch.Tensor, block_tables: torch.Tensor, block_table_stride: int,
                context_lens: torch.Tensor, max_context: int, scale: float, workspace: torch.Tensor,
                status: torch.Tensor | None = None, stream=None, overlap_previous: bool = False) -> None:
    """kv_append of one new token per sequence (position context_lens[s] - 1) fused with
    paged_decode_attention, in one launch.  overlap_previous: launch with programmatic stream
    serialization (PKV_OVERLAP_PREVIOUS; only when the kernel before it on the stream writes
    none of the lengths, tables or pool pages this step reads)."""
    desc = pool.desc if isinstance(pool, KVPool) else pool
    num_seqs, num_q_heads = int(q.shape[0]), int(q.shape[1])
    ws_bytes = workspace.numel() * workspace.element_size()
    rc = _lib.pkv_decode_step_ex(ctypes.byref(desc), _ptr(k_new), _ptr(v_new), _ptr(slot_mapping), _ptr(out),
                                 _ptr(q), num_q_heads, _ptr(block_tables), block_table_stride, _ptr(context_lens),
                                 num_seqs, max_context, scale, _ptr(workspace), ws_bytes, _ptr(status),
                                 OVERLAP_PREVIOUS if overlap_previous else 0, _stream(stream))
    _check("pkv_decode_step_ex", rc)


def paged_prefill_attention(pool: KVPool | PkvPool, out: torch.Tensor, q: torch.Tensor, query_start: torch.Tensor,
                            block_tables: torch.Tensor, block_table_stride: int, context_lens: torch.Tensor,
                            max_query: int, max_context: int, scale: float, status: torch.Tensor | None = None,
                            stream=None, overlap_previous: bool = False) -> None:
    """Causal attention of the last n_s cached tokens of each sequence (rows query_start[s] ..).
    overlap_previous: launch with PKV_OVERLAP_PREVIOUS (only when the kernel before it on the
    stream writes none of q, query_start, context_lens or block_tables, e.g. the prompt's
    kv_append)."""
    desc = pool.desc if isinstance(pool, KVPool) else pool
    num_seqs = int(context_lens.shape[0])
    rows = min(int(q.shape[0]), int(out.shape[0]))
    rc = _lib.pkv_paged_prefill_attention_ex(ctypes.byref(desc), _ptr(out), _ptr(q), int(q.shape[1]), rows,
                                             _ptr(query_start), _ptr(block_tables), block_table_stride,
                                             _ptr(context_lens), num_seqs, max_query, max_context, scale, _ptr(status),
                                             OVERLAP_PREVIOUS if overlap_previous else 0, _stream(stream))
    _check("pkv_paged_prefill_attention_ex", rc)


def paged_decode_attention_noalloc(pool: KVPool | PkvPool, out: torch.Tensor, q: torch.Tensor,
                                   block_tables: torch.Tensor, block_table_stride: int, context_lens: torch.Tensor,
                                   max_context: int, scale: float, status: torch.Tensor | None = None,
                                   stream=None) -> None:
    """paged_decode_attention without a workspace, for callers that cannot allocate device memory.

    The library keeps the split-context partial states in one fixed device array (up to
    NOALLOC_MAX_SEQS sequences) shared by every call on a device: calls must not overlap on the
    GPU, and the first call on a device should come before any stream capture there.
    """
    desc = pool.desc if isinstance(pool, KVPool) else pool
    num_seqs, num_q_heads = int(q.shape[0]), int(q.shape[1])
    rc = _lib.pkv_paged_decode_attention_noalloc(ctypes.byref(desc), _ptr(out), _ptr(q), num_q_heads,
                                                 _ptr(block_tables), block_table_stride, _ptr(context_lens),
                                                 num_seqs, max_context, scale, _ptr(status), _stream(stream))
    _check("pkv_paged_decode_attention_noalloc", rc)


class Allocator:
    """Host page allocator of ``libpkv.so`` (see ``pkv_alloc_*``): admission credits, lazy pages
    from a LIFO free list, release of a sequence's pages.  Methods raise PkvError on a negative
    status, except ``admit``, which returns the status (PKV_OK, NO_CREDIT or EXCEEDS_POOL)."""

    OK, NO_CREDIT, EXCEEDS_POOL = 0, -13, -9

    def __init__(self, num_pages: int, num_layers: int = 1, page_tokens: int = 16, max_context: int = 2048,
                 max_seqs: int = 32, free_order=None):
        import numpy as np
        self._np = np
        self.num_layers, self.max_seqs = num_layers, max_seqs
        self.max_blocks = -(-max_context // page_tokens)
        order = None
        if free_order is not None:
            self._order = np.ascontiguousarray(free_order, dtype=np.int32)
            order = self._order.ctypes.data
        h = ctypes.c_void_p()
        _check("pkv_alloc_create", _lib.pkv_alloc_create(num_pages, num_layers, page_tokens, max_context, max_seqs,
                                                         order, ctypes.byref(h)))
        self._h = h

    def __del__(self):
        h = getattr(self, "_h", None)
        if h:
            _lib.pkv_alloc_destroy(h)
            self._h = None

    def admit(self, seq: int, prompt_tokens: int, max_new_tokens: int) -> tuple[int, int]:
        """(status, credits) of admitting a request into ``seq``."""
        c = ctypes.c_int32(0)
        rc = _lib.pkv_alloc_admit(self._h, seq, prompt_tokens, max_new_tokens, ctypes.byref(c))
        if rc not in (self.OK, self.NO_CREDIT, self.EXCEEDS_POOL):
            raise PkvError("pkv_alloc_admit", rc)
        return rc, c.value

    def page(self, seq: int, layer: int, block: int) -> int:
        p = ctypes.c_int32(-1)
        _check("pkv_alloc_page", _lib.pkv_alloc_page(self._h, seq, layer, block, ctypes.byref(p)))
        return p.value

    def free_seq(self, seq: int) -> None:
        _check("pkv_alloc_free_seq", _lib.pkv_alloc_free_seq(self._h, seq))

    def block_tables(self):
        """A copy of the block table [max_seqs, num_layers, max_blocks]."""
        n = self.max_seqs * self.num_layers * self.max_blocks
        ptr = _lib.pkv_alloc_block_tables(self._h)
        return self._np.ctypeslib.as_array(ptr, shape=(n,)).copy().reshape(self.max_seqs, self.num_layers,
                                                                           self.max_blocks)

    def state(self) -> tuple[int, int]:
        """(free pages, credits in use)."""
        f, c = ctypes.c_int32(0), ctypes.c_int32(0)
        _check("pkv_alloc_state", _lib.pkv_alloc_state(self._h, ctypes.byref(f), ctypes.byref(c)))
        return f.value, c.value


class Scheduler:
    """Host page allocator + continuous-batching scheduler of ``libpkv.so`` (see ``pkv_sched_*``)."""

    def __init__(self, num_pages: int, num_layers: int = 1, page_tokens: int = 16, max_context: int = 2048,
                 num_slots: int = 32, free_order=None):
        import numpy as np
        self._np = np
        self.num_layers, self.num_slots = num_layers, num_slots
        order = None
        if free_order is not None:
            self._order = np.ascontiguousarray(free_order, dtype=np.int32)
            order = self._order.ctypes.data
        h = ctypes.c_void_p()
        _check("pkv_sched_create", _lib.pkv_sched_create(num_pages, num_layers, page_tokens, max_context, num_slots,
                                                         order, ctypes.byref(h)))
        self._h = h

    def __del__(self):
        h = getattr(self, "_h", None)
        if h:
            _lib.pkv_sched_destroy(h)
            self._h = None

    def submit(self, request_id: int, prompt_tokens: int, max_new_tokens: int) -> None:
        _check("pkv_sched_submit", _lib.pkv_sched_submit(self._h, int(request_id), int(prompt_tokens),
                                                         int(max_new_tokens)))

    def step(self) -> dict:
        """One step; returns copies of the plan as numpy arrays."""
        np = self._np
        plan = PkvStepPlan()
        _check("pkv_sched_step", _lib.pkv_sched_step(self._h, ctypes.byref(plan)))

        def arr(ptr, n, dt):
            if n == 0:
                return np.zeros(0, dtype=dt)
            return np.ctypeslib.as_array(ptr, shape=(n,)).astype(dt, copy=True)

        na, L, S = plan.num_appends, self.num_layers, self.num_slots
        return {
            "finished": arr(plan.finished_request, plan.num_finished, np.int64),
            "admitted": arr(plan.admitted_request, plan.num_admitted, np.int64),
            "admitted_slot": arr(plan.admitted_slot, plan.num_admitted, np.int32),
            "append_request": arr(plan.append_request, na, np.int64),
            "append_position": arr(plan.append_position, na, np.int32),
            "append_slot_mapping": arr(plan.append_slot_mapping, na * L, np.int32).reshape(L, na),
            "decode_slot": arr(plan.decode_slot, plan.num_decode, np.int32),
            "context_lens": arr(plan.context_lens, S, np.int32),
            "block_tables": arr(plan.block_tables, S * L * plan.max_blocks, np.int32).reshape(S, L, plan.max_blocks),
        }

    def stats(self) -> dict:
        st = PkvSchedStats()
        _check("pkv_sched_stats_get", _lib.pkv_sched_stats_get(self._h, ctypes.byref(st)))
        return {name: int(getattr(st, name)) for name, _ in PkvSchedStats._fields_}
