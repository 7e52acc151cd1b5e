"""The allocation-free decode entry point gives the same results as the regular one.

Some callers cannot allocate device memory - a plugin inside a runtime that owns
every device buffer, or a C/FFI caller without an allocator of its own that must
not call cudaMalloc in the middle of a run - so pkv_paged_decode_attention_noalloc
keeps its split-context partial states in a fixed array inside the library instead
of a caller workspace.  This file is collected last; it passes both alone in a
fresh process and after the other tests (the fixed array keeps whatever an earlier
call left in it, and nothing in it has to start at zero).
"""
import pytest
import torch

from tests import gpu_util as U
from workloads import configs

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _gpu():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")


def _both(d: U.DeviceDecode):
    """Output of the regular entry point (with a workspace) and of the allocation-free one."""
    import paged_kv_cache_180_gb300 as pkv
    wl = d.wl
    q = d.q(0)
    ref = d.attend(0, q=q).clone()
    out = torch.full_like(ref, float("nan"))
    pkv.paged_decode_attention_noalloc(d.pool, out, q, d.bt.view(-1), wl.num_layers * wl.max_blocks, d.lens,
                                       wl.max_context, wl.scale, d.status)
    torch.cuda.synchronize()
    return ref.cpu().double().numpy(), out.cpu().double().numpy()


def test_noalloc_matches_workspace_entry_point_on_two_calls_in_a_row():
    first = configs.ragged(seed=900, num_seqs=64)
    second = configs.custom(901, [2048, 1, 700, 33, 0, 1500, 16], name="second")
    for wl in (first, second):
        d = U.DeviceDecode(wl)
        d.append_all()
        ref, got = _both(d)
        U.assert_close(got, ref, f"noalloc vs workspace ({wl.name})")
        assert d.status_value() == 0


def test_noalloc_rejects_more_sequences_than_its_scratch_holds():
    import paged_kv_cache_180_gb300 as pkv
    n = pkv.binding.NOALLOC_MAX_SEQS + 1
    wl = configs.custom(902, [1] * n, name="too_many")
    d = U.DeviceDecode(wl)
    with pytest.raises(pkv.PkvError) as e:
        pkv.paged_decode_attention_noalloc(d.pool, d.out, d.q(0), d.bt.view(-1), wl.max_blocks, d.lens,
                                           wl.max_context, wl.scale, d.status)
    assert e.value.code == -12  # PKV_ERR_NOALLOC_LIMIT; nothing was enqueued
