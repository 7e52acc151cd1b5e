"""Paged BF16 KV-cache decode attention for GB300 (sm_103a).

The compute path is the C-ABI library ``libpkv.so`` (hand-written CUDA kernels,
declared in ``include/pkv.h``); ``binding`` is its thin Python wrapper.  Build the
library with ``python -m paged_kv_cache_180_gb300.build``.

The public names below load the binding on first use; if ``libpkv.so`` is
missing that raises ImportError (there is no fallback path).
"""
_PUBLIC = ("KVPool", "PkvError", "PkvPool", "decode_max_ctas", "decode_plan", "decode_step", "decode_workspace", "decode_workspace_bytes",
           "kv_append", "kv_pool_bytes", "kv_pool_create", "paged_decode_attention",
           "paged_decode_attention_noalloc", "paged_prefill_attention", "Scheduler", "Allocator",
           "status_string")


def __getattr__(name):
    if name in _PUBLIC or name == "binding":
        import importlib
        binding = importlib.import_module(__name__ + ".binding")
        return binding if name == "binding" else getattr(binding, name)
    raise AttributeError(name)


__all__ = list(_PUBLIC)
