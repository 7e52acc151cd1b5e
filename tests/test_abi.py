"""The C-ABI library loads, exports every symbol include/pkv.h declares, and checks its
arguments on the host (no GPU needed: none of these calls reaches a kernel launch)."""
import ctypes
import os
import re

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "pkv.h")


@pytest.fixture(scope="module")
def binding():
    from paged_kv_cache_180_gb300 import build
    build.build()
    from paged_kv_cache_180_gb300 import binding as b
    return b


def declared_functions():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(pkv_\w+)\s*\(", text)))


def test_header_declares_the_boundary():
    names = declared_functions()
    for required in ("pkv_kv_pool_create", "pkv_kv_append", "pkv_paged_decode_attention",
                     "pkv_decode_workspace_bytes", "pkv_status_string"):
        assert required in names


def test_every_declared_symbol_is_exported(binding):
    lib = ctypes.CDLL(binding.LIB_PATH)
    missing = [n for n in declared_functions() if not hasattr(lib, n)]
    assert not missing, missing
    assert set(declared_functions()) <= set(binding.EXPORTS), "binding lacks a declared entry point"


def test_pool_bytes_and_create_validation(binding):
    b = binding
    assert b.kv_pool_bytes(4096) == 128 * 1024 * 1024          # 128 MiB = 4096 pages of 32 KiB
    assert b.kv_pool_bytes(0) == 0
    base = 1 << 20   # a fake, aligned device address: create never dereferences it
    d = b.kv_pool_create(base, base + 16384, 0, 8)
    assert d.page_stride_bytes == 32768 and d.num_pages == 8
    for args, code in [((base + 8, base + 16384, 0, 8), -4), ((base, base + 16384, 0, 8, 16, 8, 128), -3),
                       ((base, base + 16384, 0, 0), -2), ((0, base, 0, 8), -1), ((base, base + 16384, 100, 8), -2),
                       ((base, base + 16384, 32776, 8), -4)]:
        with pytest.raises(b.PkvError) as e:
            b.kv_pool_create(*args)
        assert e.value.code == code, (args, e.value.code)


def test_decode_host_checks_return_before_any_launch(binding):
    b = binding
    lib = b._lib
    base = 1 << 20
    d = b.kv_pool_create(base, base + 16384, 0, 8)
    ws = b.decode_workspace_bytes(4)
    assert ws > 0 and b.decode_workspace_bytes(4, 16, 64) == 0
    P = ctypes.c_void_p
    # unsupported head count, null pointers, bad scale, small workspace, misalignment
    call = lambda **kw: lib.pkv_paged_decode_attention(  # noqa: E731
        ctypes.byref(d), P(kw.get("out", base)), P(kw.get("q", base)), kw.get("hq", 32), P(base), 128, P(base),
        kw.get("n", 4), 2048, kw.get("scale", 0.125), P(kw.get("ws", base)), kw.get("wsb", ws), None, None)
    assert call(hq=16) == -3
    assert call(q=0) == -1
    assert call(scale=float("inf")) == -5
    assert call(wsb=ws - 1) == -6
    assert call(q=base + 2) == -4
    assert call(n=0) == 0                  # nothing to do
    assert call(n=-1) == -2
    assert lib.pkv_kv_append(ctypes.byref(d), P(base), P(base), P(base), 0, None, None) == 0
    assert lib.pkv_kv_append(ctypes.byref(d), P(base + 4), P(base), P(base), 1, None, None) == -4
    assert lib.pkv_kv_append(ctypes.byref(d), None, P(base), P(base), 1, None, None) == -1
    # decode_step_ex: unknown flag bits are refused before anything else; a null new-row
    # pointer with a known flag is caught by the pointer checks
    step = lambda flags, k=base: lib.pkv_decode_step_ex(  # noqa: E731
        ctypes.byref(d), P(k), P(base), P(base), P(base), P(base), 32, P(base), 128, P(base), 4, 2048, 0.125,
        P(base), ws, None, flags, None)
    assert step(2) == -2
    assert step(b.OVERLAP_PREVIOUS, k=0) == -1
    # prefill_ex: unknown flag bits refused first; a null output with a known flag is caught
    pre = lambda flags, out=base: lib.pkv_paged_prefill_attention_ex(  # noqa: E731
        ctypes.byref(d), P(out), P(base), 32, 64, P(base), P(base), 128, P(base), 4, 16, 2048, 0.125, None, flags,
        None)
    assert pre(4) == -2
    assert pre(b.OVERLAP_PREVIOUS, out=0) == -1


def test_status_strings(binding):
    for code in range(-13, 1):
        assert binding.status_string(code) != "unknown status"
    assert binding.status_string(-99) == "unknown status"


def test_workspace_size_formula(binding):
    # (max CTAs + num_seqs) slots of 32 heads x (64 acc + (m, l)) floats + 2 x 8 ticket counters
    n = 256
    slots = binding.decode_max_ctas() + n
    assert binding.decode_workspace_bytes(n) == slots * (32 * 64 * 4 + 32 * 8 + 2 * 8 * 4)


def test_plan_without_gpu_is_bounded(binding):
    g, launches = binding.decode_plan(256, 2048)
    assert 1 <= g <= binding.decode_max_ctas() and launches == 1
    g, _ = binding.decode_plan(1, 17)
    assert g == 1
