"""Paged BF16 KV-cache decode attention for GB300 (sm_103a).

The compute path is the C-ABI library ``libpkv.so`` (hand-written CUDA kernels,
declared in ``include/pkv.h``); ``binding`` is its thin Python wrapper.  Build the
library with ``python -m paged_kv_cache_180_gb300.build``.
"""
from . import binding  # noqa: F401  (fails loudly when libpkv.so is missing)
from .binding import (KVPool, decode_max_ctas, decode_plan, decode_workspace_bytes, kv_append,  # noqa: F401
                      kv_pool_bytes, kv_pool_create, paged_decode_attention, status_string)
