"""The allocation-free decode entry point gives the results of the regular one and of the oracle.

Some callers cannot allocate device memory - a plugin inside a runtime that owns
every device buffer, or a C/FFI caller without an allocator of its own that must
not call cudaMalloc in the middle of a run - so pkv_paged_decode_attention_noalloc
keeps its split-context partial states in a fixed array inside the library instead
of a caller workspace.  Its merge counters must start at zero: the first call on a
device clears the array on that call's stream.  This file is collected last; it
passes both alone in a fresh process and after the other tests (the array keeps
whatever the last call left in it).
"""
import os
import subprocess
import sys
import textwrap

import pytest
import torch

import oracle
from tests import gpu_util as U
from workloads import configs

pytestmark = pytest.mark.gpu

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module", autouse=True)
def _gpu():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")


def _both(d: U.DeviceDecode, stream=None):
    """Output of the regular entry point (with a workspace) and of the allocation-free one."""
    import paged_kv_cache_180_gb300 as pkv
    wl = d.wl
    q = d.q(0)
    ref = d.attend(0, q=q).clone()
    out = torch.full_like(ref, float("nan"))
    pkv.paged_decode_attention_noalloc(d.pool, out, q, d.bt.view(-1), wl.num_layers * wl.max_blocks, d.lens,
                                       wl.max_context, wl.scale, d.status, stream=stream)
    torch.cuda.synchronize()
    return ref.cpu().double().numpy(), out.cpu().double().numpy()


def test_noalloc_matches_workspace_entry_point_and_oracle_on_two_calls_in_a_row():
    first = configs.ragged(seed=900, num_seqs=64)
    second = configs.custom(901, [2048, 1, 700, 33, 0, 1500, 16], name="second")
    for wl in (first, second):
        d = U.DeviceDecode(wl)
        d.append_all()
        ref, got = _both(d)
        U.assert_close(got, ref, f"noalloc vs workspace ({wl.name})")
        expect, err, _ = oracle.decode_workload(wl)
        assert err == 0
        U.assert_close(got, expect, f"noalloc vs oracle ({wl.name})")
        assert d.status_value() == 0


def test_noalloc_at_its_largest_batch():
    """PKV_NOALLOC_MAX_SEQS sequences (mixed lengths, so the split cuts sequences and uses the
    merge slots of all of them) in one call, then a second call of the same size."""
    import paged_kv_cache_180_gb300 as pkv
    n = pkv.binding.NOALLOC_MAX_SEQS
    for seed in (903, 904):
        wl = configs.custom(seed, [1 + (37 * i + seed) % 400 for i in range(n)], name=f"max_batch_{seed}")
        d = U.DeviceDecode(wl)
        d.append_all()
        ref, got = _both(d)
        U.assert_close(got, ref, f"noalloc vs workspace, {n} sequences")
        expect, err = U.oracle_decode_threaded(wl)
        assert err == 0
        U.assert_close(got, expect, f"noalloc vs oracle, {n} sequences")
        assert d.status_value() == 0


_FRESH_PROCESS = textwrap.dedent("""
    import sys
    import numpy as np
    import torch
    sys.path.insert(0, {root!r})
    import paged_kv_cache_180_gb300 as pkv
    from tests import gpu_util as U
    from workloads import configs
    torch.cuda.init()
    wl = configs.ragged(seed=905, num_seqs=96)
    side = torch.cuda.Stream()        # torch side streams are non-blocking
    with torch.cuda.stream(side):
        d = U.DeviceDecode(wl)
        d.append_all()
        q = d.q(0)
        out = torch.full((wl.num_seqs, 32, 64), float("nan"), dtype=torch.float32, device=U.dev())
        # the first allocation-free call of this process, on the side stream
        pkv.paged_decode_attention_noalloc(d.pool, out, q, d.bt.view(-1), wl.max_blocks, d.lens, wl.max_context,
                                           wl.scale, d.status, stream=side)
        ref = d.attend(0, q=q)
    side.synchronize()
    assert int(d.status.item()) == 0
    U.assert_close(out.cpu().double().numpy(), ref.cpu().double().numpy(), "first call on a side stream")
    print("fresh-process side-stream call ok")
""")


def test_first_call_in_a_fresh_process_on_a_side_stream():
    """The first call's clear of the array is ordered before its kernel on the caller's own
    (non-blocking) stream."""
    r = subprocess.run([sys.executable, "-c", _FRESH_PROCESS.format(root=ROOT)], cwd=ROOT, capture_output=True,
                       text=True, timeout=600)
    assert r.returncode == 0, r.stdout + r.stderr
    assert "side-stream call ok" in r.stdout


def test_noalloc_rejects_more_sequences_than_its_scratch_holds():
    import paged_kv_cache_180_gb300 as pkv
    n = pkv.binding.NOALLOC_MAX_SEQS + 1
    wl = configs.custom(902, [1] * n, name="too_many")
    d = U.DeviceDecode(wl)
    with pytest.raises(pkv.PkvError) as e:
        pkv.paged_decode_attention_noalloc(d.pool, d.out, d.q(0), d.bt.view(-1), wl.max_blocks, d.lens,
                                           wl.max_context, wl.scale, d.status)
    assert e.value.code == -12  # PKV_ERR_NOALLOC_LIMIT; nothing was enqueued
