"""GPU parity of paged prefill attention (through the C ABI) against the oracle.

Full prefills (the whole context is the query chunk), chunked prefills (a cached
prefix plus a chunk), single queries (decode through the prefill entry point),
ragged mixes in one launch, lengths not multiples of the 32-token tile or the
16-token page, stale NaN bytes past each context, invalid sequences, the first query
of a fresh prefill returning V[0] exactly, and page-permutation bit-exactness.
Tolerance |gpu - oracle| <= 1e-3 + 1e-2 |oracle|.
"""
import numpy as np
import pytest
import torch

import oracle
from tests import gpu_util as U
from workloads import configs, rng

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _gpu():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")


def _run(wl, nq, seed=1, bt=None, scale=None):
    """Queries = the last nq[s] tokens of each sequence (all already appended)."""
    scale = wl.scale if scale is None else scale
    import paged_kv_cache_180_gb300 as pkv
    d = U.DeviceDecode(wl)
    d.append_all()
    qs = np.concatenate([[0], np.cumsum(nq)]).astype(np.int32)
    total = int(qs[-1])
    qbits = rng.normal_bf16(rng.stream_key(seed, "pf-q"), 0, total * 32 * 64).reshape(total, 32, 64)
    out = torch.full((max(total, 1), 32, 64), float("nan"), dtype=torch.float32, device=U.dev())
    bt_host = np.ascontiguousarray(wl.block_tables[:, 0, :] if bt is None else bt)
    pkv.paged_prefill_attention(d.pool, out, U.to_dev(qbits), U.to_dev(qs), U.to_dev(bt_host), bt_host.shape[1],
                                d.lens, max(max(nq), 1), wl.max_context, scale, d.status)
    got = out[:total].cpu().double().numpy()
    opool = oracle.Pool(wl.num_pages)
    k, v, slots = wl.kv_all(0)
    oracle.kv_append(opool, k, v, slots)
    ref, err = oracle.paged_prefill_attention(opool, qbits, qs, bt_host, wl.context_lens, scale, wl.max_context)
    return got, ref, err, d.status_value(), qs


def test_full_prefills():
    wl = configs.custom(600, [512, 17, 64, 100, 1], name="full")
    nq = [512, 17, 64, 100, 1]
    got, ref, err, st, _ = _run(wl, nq)
    assert err == 0 and st == 0
    U.assert_close(got, ref, "full prefill")


def test_chunked_prefills_and_single_queries():
    wl = configs.custom(601, [2048, 700, 33, 1000, 16, 5], name="chunked")
    nq = [128, 1, 33, 77, 16, 2]
    got, ref, err, st, _ = _run(wl, nq)
    assert err == 0 and st == 0
    U.assert_close(got, ref, "chunked prefill")


def test_llama_prompt_shapes():
    # prompts of the Llama step: 4 sequences, the whole context as the chunk (ctx up to 2048)
    wl = configs.custom(602, [128, 512, 1024, 2048], name="llama_prefill")
    got, ref, err, st, _ = _run(wl, [128, 512, 1024, 2048])
    assert err == 0 and st == 0
    U.assert_close(got, ref, "llama prompts")


def test_first_query_of_fresh_prefill_is_v0_exactly():
    wl = configs.custom(603, [40, 3], name="v0")
    got, ref, err, st, qs = _run(wl, [40, 3])
    for s in range(2):
        _, v = wl.kv_tokens(s)
        want = np.repeat(rng.bf16_bits_to_f64(v[0]), 4, axis=0).astype(np.float32)
        assert np.array_equal(got[qs[s]].astype(np.float32), want)


def test_invalid_sequences():
    wl = configs.custom(604, [10, 30, 2049], num_pages=8, name="bad")
    got, ref, err, st, qs = _run(wl, [11, 4, 3])    # 11 queries > 10 cached; 2049 > max_context
    assert st == 2
    assert not got[:11].any() and not got[15:].any()
    U.assert_close(got[11:15], ref[11:15], "valid sequence beside invalid ones")


def test_page_permutation_bit_exact():
    wl = configs.custom(605, [300, 90], name="perm")
    got1, _, _, _, _ = _run(wl, [60, 90])
    perm = rng.permutation(rng.stream_key(606, "move"), wl.num_pages)
    bt2 = np.where(wl.block_tables >= 0, perm[np.maximum(wl.block_tables, 0)], -1).astype(np.int32)
    wl2 = configs.DecodeWorkload(wl.name, wl.seed, wl.num_pages, 1, wl.context_lens, bt2)
    got2, _, _, _, _ = _run(wl2, [60, 90])
    assert np.array_equal(got1.astype(np.float32).view(np.int32), got2.astype(np.float32).view(np.int32))


@pytest.mark.parametrize("scale", [1.0, -1.0, -0.125, 0.0])
def test_scales_moving_max_and_sign(scale):
    # scale 1: scores spread ~8x wider than at 1/sqrt(64), so a row's running maximum
    # jumps by more than 2^8 after its first key block and the kernel must rescale O and
    # the row sum; negative scales flip which keys dominate; scale 0 is a uniform average
    wl = configs.custom(607, [700, 300, 64], name="scales")
    got, ref, err, st, _ = _run(wl, [700, 150, 64], scale=scale)
    assert err == 0 and st == 0
    U.assert_close(got, ref, f"scale {scale}")


def test_invalid_page_inside_a_span():
    # a block-table entry past the pool inside sequence 0's span: the device flags it and
    # leaves that page out (finite rows); the other sequence of the launch is unaffected
    wl = configs.custom(608, [200, 90], name="badpage")
    bt = np.ascontiguousarray(wl.block_tables[:, 0, :]).copy()
    bt[0, 5] = wl.num_pages + 7
    got, ref, err, st, qs = _run(wl, [64, 90], bt=bt)
    assert st & 4 and err & 4
    assert np.isfinite(got[qs[0]:qs[1]]).all()
    U.assert_close(got[qs[1]:qs[2]], ref[qs[1]:qs[2]], "sequence beside the invalid page")


def test_query_rows_past_the_buffers():
    # q and out one row shorter than query_start says: the last sequence counts as invalid
    # (status bit, nothing read or written past the buffers); the other one is exact
    import paged_kv_cache_180_gb300 as pkv
    wl = configs.custom(609, [300, 70], name="short_rows")
    nq = [100, 40]
    d = U.DeviceDecode(wl)
    d.append_all()
    qs = np.array([0, 100, 140], dtype=np.int32)
    qbits = rng.normal_bf16(rng.stream_key(2, "pf-q"), 0, 140 * 32 * 64).reshape(140, 32, 64)
    q = U.to_dev(qbits)[:139]
    out = torch.full((139, 32, 64), float("nan"), dtype=torch.float32, device=U.dev())
    bt_host = np.ascontiguousarray(wl.block_tables[:, 0, :])
    pkv.paged_prefill_attention(d.pool, out, q, U.to_dev(qs), U.to_dev(bt_host), bt_host.shape[1], d.lens, 100,
                                wl.max_context, wl.scale, d.status)
    got = out.cpu().double().numpy()
    assert d.status_value() & 2
    opool = oracle.Pool(wl.num_pages)
    k, v, slots = wl.kv_all(0)
    oracle.kv_append(opool, k, v, slots)
    ref, err = oracle.paged_prefill_attention(opool, qbits, qs, bt_host, wl.context_lens, wl.scale, wl.max_context)
    U.assert_close(got[:100], ref[:100], "sequence inside the buffers")
    assert not got[100:].any()


def test_prefill_overlapping_the_append():
    """The prompt's K/V appended by kv_append into a pool of NaN bytes, and the prefill launched
    right after it with overlap_previous: its set-up may run during the append, but its page
    reads come after it (a page read early would bring NaN into the output)."""
    import paged_kv_cache_180_gb300 as pkv
    wl = configs.custom(612, [512, 300, 1000, 64, 2048], name="overlap")
    nq = [512, 300, 200, 64, 1]
    d = U.DeviceDecode(wl)  # pool filled with a NaN pattern
    k, v, slots = (U.to_dev(a) for a in wl.kv_all(0))
    qs = np.concatenate([[0], np.cumsum(nq)]).astype(np.int32)
    total = int(qs[-1])
    qbits = rng.normal_bf16(rng.stream_key(612, "pf-q"), 0, total * 32 * 64).reshape(total, 32, 64)
    q, qs_d = U.to_dev(qbits), U.to_dev(qs)
    bt_host = np.ascontiguousarray(wl.block_tables[:, 0, :])
    bt = U.to_dev(bt_host)
    out = torch.full((total, 32, 64), float("nan"), dtype=torch.float32, device=U.dev())
    torch.cuda.synchronize()
    pkv.kv_append(d.pool, k, v, slots, d.status)
    pkv.paged_prefill_attention(d.pool, out, q, qs_d, bt, bt_host.shape[1], d.lens, max(nq), wl.max_context,
                                wl.scale, d.status, overlap_previous=True)
    assert d.status_value() == 0
    opool = oracle.Pool(wl.num_pages)
    oracle.kv_append(opool, *wl.kv_all(0))
    ref, err = oracle.paged_prefill_attention(opool, qbits, qs, bt_host, wl.context_lens, wl.scale, wl.max_context)
    assert err == 0
    U.assert_close(out.cpu().double().numpy(), ref, "prefill overlapping the append")


def test_max_query_bound_leaves_longer_runs_alone():
    """max_query sizes the grid: only the first max_query query rows of each sequence are
    computed (exactly); rows past it are not written."""
    import paged_kv_cache_180_gb300 as pkv
    wl = configs.custom(613, [300, 90, 40], name="maxq")
    nq = [100, 90, 20]
    d = U.DeviceDecode(wl)
    d.append_all()
    qs = np.concatenate([[0], np.cumsum(nq)]).astype(np.int32)
    total = int(qs[-1])
    qbits = rng.normal_bf16(rng.stream_key(613, "pf-q"), 0, total * 32 * 64).reshape(total, 32, 64)
    out = torch.full((total, 32, 64), float("nan"), dtype=torch.float32, device=U.dev())
    bt_host = np.ascontiguousarray(wl.block_tables[:, 0, :])
    pkv.paged_prefill_attention(d.pool, out, U.to_dev(qbits), U.to_dev(qs), U.to_dev(bt_host), bt_host.shape[1],
                                d.lens, 32, wl.max_context, wl.scale, d.status)
    assert d.status_value() == 0
    got = out.cpu().double().numpy()
    opool = oracle.Pool(wl.num_pages)
    oracle.kv_append(opool, *wl.kv_all(0))
    ref, err = oracle.paged_prefill_attention(opool, qbits, qs, bt_host, wl.context_lens, wl.scale, wl.max_context)
    assert err == 0
    for s in range(3):
        done = min(nq[s], 32)
        rows = slice(int(qs[s]), int(qs[s]) + done)
        U.assert_close(got[rows], ref[rows], f"sequence {s}, first {done} queries")
        assert np.isnan(got[int(qs[s]) + done:int(qs[s + 1])]).all()
