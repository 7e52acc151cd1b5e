"""GPU parity of the CUDA path (through the C ABI) against the CPU oracle.

* kv_append and block-table indexing: bit-exact pool bytes.
* Attention: |gpu - oracle| <= 1e-3 + 1e-2 |oracle| elementwise, FP32 output vs FP64 oracle.
* Invariants on the GPU: physical page order does not change a single bit, a
  one-token context returns V exactly, the result does not depend on the split
  count beyond rounding, empty and invalid inputs give zero rows and status bits.
"""
import math

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
    import paged_kv_cache_180_gb300  # noqa: F401  (fails loudly without libpkv.so)


def _oracle_pool_bytes(opool: oracle.Pool) -> np.ndarray:
    return opool.data.reshape(-1)


# ---------------------------------------------------------------------------
@pytest.mark.parametrize("make", [configs.tiny, lambda: configs.ragged(num_seqs=16)], ids=["tiny", "ragged16"])
def test_append_bit_exact(make):
    wl = make()
    d = U.DeviceDecode(wl)
    d.append_all()
    assert d.status_value() == 0
    opool = oracle.Pool(wl.num_pages)
    k, v, slots = wl.kv_all(0)
    assert oracle.kv_append(opool, k, v, slots) == 0
    got = U.bits(d.pool.view()).reshape(-1)
    np.testing.assert_array_equal(got, _oracle_pool_bytes(opool))


def test_append_decode_token_and_padding_slots():
    wl = configs.ragged(seed=300, num_seqs=8)
    d = U.DeviceDecode(wl)
    d.append_all()
    # overwrite every sequence's last token with fresh values, with padding slots mixed in
    kn, vn, sn = wl.decode_tokens(0)
    r = np.random.default_rng(5)
    kn = rng.f64_to_bf16_bits(r.standard_normal(kn.shape))
    vn = rng.f64_to_bf16_bits(r.standard_normal(vn.shape))
    sn = sn.copy()
    sn[::3] = -1
    d.pkv.kv_append(d.pool, U.to_dev(kn), U.to_dev(vn), U.to_dev(sn), d.status)
    assert d.status_value() == 0
    opool = oracle.Pool(wl.num_pages)
    k, v, slots = wl.kv_all(0)
    oracle.kv_append(opool, k, v, slots)
    oracle.kv_append(opool, kn, vn, sn)
    np.testing.assert_array_equal(U.bits(d.pool.view()).reshape(-1), _oracle_pool_bytes(opool))


def test_append_bad_slot_sets_status_and_skips():
    wl = configs.tiny()
    d = U.DeviceDecode(wl)
    before = U.bits(d.pool.view()).copy()
    k = U.to_dev(np.zeros((2, 8, 64), np.uint16))
    slots = U.to_dev(np.array([wl.num_pages * 16, -5], np.int32))
    d.pkv.kv_append(d.pool, k, k, slots, d.status)
    assert d.status_value() == 1  # PKV_DEV_BAD_SLOT
    np.testing.assert_array_equal(U.bits(d.pool.view()), before)


# ---------------------------------------------------------------------------
def _check_workload(wl, layers=(0,), num_ctas=0, seqs=None):
    d = U.DeviceDecode(wl)
    for layer in layers:
        d.append_all(layer)
    worst = 0.0
    for layer in layers:
        out = d.attend(layer, num_ctas=num_ctas).cpu().double().numpy()
        ref, err, _ = oracle.decode_workload(wl, layer=layer)
        assert err == 0
        worst = max(worst, U.assert_close(out, ref, f"{wl.name} layer {layer}"))
    assert d.status_value() == 0
    return worst


def test_tiny_parity():
    _check_workload(configs.tiny())


def test_ragged_parity():
    _check_workload(configs.ragged())


def test_llama_step_all_layers_parity():
    # 16 layers share one 4096-page pool; the table of layer l is passed as base + l*128, stride 16*128
    _check_workload(configs.llama_step(), layers=range(16))


@pytest.mark.parametrize("num_ctas", [1, 2, 3, 7, 31, 64, 150, 304, 1024])
def test_split_count_sweep(num_ctas):
    # more CTAs than pages (1024 > 187) leaves empty CTAs inside a sequence's span
    wl = configs.custom(401, [1, 17, 300, 2048, 16, 33, 512, 5], name="sweep")
    _check_workload(wl, num_ctas=num_ctas)


def test_page_permutation_bit_exact():
    wl = configs.ragged(seed=410, num_seqs=12)
    d1 = U.DeviceDecode(wl)
    d1.append_all()
    out1 = d1.attend(num_ctas=37).clone()
    perm = rng.permutation(rng.stream_key(411, "move"), wl.num_pages)   # old page id -> new
    bt2 = np.where(wl.block_tables >= 0, perm[np.maximum(wl.block_tables, 0)], -1).astype(np.int32)
    wl2 = configs.DecodeWorkload(wl.name, wl.seed, wl.num_pages, wl.num_layers, wl.context_lens, bt2)
    d2 = U.DeviceDecode(wl2)
    d2.append_all()
    out2 = d2.attend(num_ctas=37)
    assert torch.equal(out1.view(torch.int32), out2.view(torch.int32))
    assert d1.status_value() == 0 and d2.status_value() == 0


def test_one_token_context_returns_v_exactly():
    wl = configs.custom(420, [1, 1, 1, 1, 1, 1, 1, 1, 1, 1], name="one")
    d = U.DeviceDecode(wl)
    d.append_all()
    out = d.attend().cpu().numpy()
    for s in range(wl.num_seqs):
        _, v = wl.kv_tokens(s)
        want = np.repeat(rng.bf16_bits_to_f64(v[0]), 4, axis=0).astype(np.float32)
        assert np.array_equal(out[s], want)


def test_identical_keys_give_mean_of_v():
    wl = configs.custom(430, [100, 37], name="samekeys")
    d = U.DeviceDecode(wl)
    ks, vs, ss = [], [], []
    r = np.random.default_rng(3)
    for s in range(wl.num_seqs):
        c = int(wl.context_lens[s])
        key = rng.f64_to_bf16_bits(r.standard_normal((1, 8, 64)))
        ks.append(np.repeat(key, c, axis=0))
        vs.append(wl.kv_tokens(s)[1])
        ss.append(wl.slot_mapping(s, 0, 0, c))
    d.pkv.kv_append(d.pool, U.to_dev(np.concatenate(ks)), U.to_dev(np.concatenate(vs)),
                    U.to_dev(np.concatenate(ss)), d.status)
    out = d.attend(num_ctas=3).cpu().double().numpy()
    for s in range(wl.num_seqs):
        mean_v = np.repeat(rng.bf16_bits_to_f64(vs[s]).mean(axis=0), 4, axis=0)
        U.assert_close(out[s], mean_v, "mean of V")


def test_spiky_scores_parity():
    # 1 % of K entries scaled x8 (as the 16-layer config) plus one key aligned with its query
    wl = configs.custom(440, [700, 64, 1500], spike_prob=0.01, name="spiky")
    _check_workload(wl, num_ctas=5)


def test_empty_and_invalid_contexts():
    wl = configs.custom(450, [0, 40, 2049, 16, -3, 1], num_pages=16, name="edge")
    d = U.DeviceDecode(wl)
    d.append_all(seqs=[1, 3, 5])
    d.out.fill_(7.0)
    out = d.attend(max_context=2048).cpu().double().numpy()
    assert d.status_value() == 2  # PKV_DEV_BAD_CONTEXT
    ref, err, _ = oracle.decode_workload(wl, seqs=[1, 3, 5])
    for s in (0, 2, 4):
        assert not out[s].any()
    U.assert_close(out[[1, 3, 5]], ref[[1, 3, 5]], "edge")


def test_batch_without_pages_gives_zero_rows():
    # no sequence has a page (contexts 0, or invalid): no CTA walks pages, every row is zero
    for lens, status in (([0, 0, 0], 0), ([0, -5, 3000], 2)):
        wl = configs.custom(452, lens, num_pages=4, name="nopages")
        d = U.DeviceDecode(wl)
        d.out.fill_(7.0)
        out = d.attend(max_context=2048).cpu().double().numpy()
        assert not out.any()
        assert d.status_value() == status


# Grids small enough for clusters of 8 (one CTA per SM) merge a cut sequence's parts on chip,
# and only sequences cut across clusters meet in the workspace.  These splits put a
# sequence's parts in one cluster (2 .. 8 CTAs: every receive-slot layout), across two or
# more clusters (level-two tickets), and a single part in a cluster at either end.
@pytest.mark.parametrize("lens,num_ctas", [
    ([2048], 2), ([2048], 5), ([2048], 7), ([2048], 8), ([2048], 9), ([2048], 17), ([2048], 63),
    ([2048], 120), ([128, 512, 1024, 2048], 58), ([128, 512, 1024, 2048], 0), ([300, 7, 1500, 40, 900], 13),
    ([300, 7, 1500, 40, 900], 0), ([16] * 40 + [2048], 33)])
def test_cluster_merge_layouts(lens, num_ctas):
    wl = configs.custom(455, lens, spike_prob=0.01, name=f"clusters-{len(lens)}-{num_ctas}")
    _check_workload(wl, num_ctas=num_ctas)


def test_small_grids_launch_in_whole_clusters():
    import paged_kv_cache_180_gb300 as pkv
    g, _ = pkv.decode_plan(4, 2048)   # the Llama-shaped batch: a grid of whole 8-CTA clusters
    assert g % 8 == 0 and 8 <= g <= 152
    g, _ = pkv.decode_plan(256, 2048)  # a large batch: two CTAs per SM, no clusters
    assert g > 152


def test_invalid_page_sets_status_and_stays_finite():
    wl = configs.custom(460, [48, 20], name="badpage")
    d = U.DeviceDecode(wl)
    d.append_all()
    bt = wl.block_tables.copy()
    bt[0, 0, 1] = wl.num_pages + 3
    d.bt = U.to_dev(bt)
    out = d.attend().cpu().double().numpy()
    assert d.status_value() == 4  # PKV_DEV_BAD_PAGE
    assert np.isfinite(out).all()
    ref, err, _ = oracle.decode_workload(wl)
    U.assert_close(out[1], ref[1], "untouched sequence")


def test_workspace_reuse_and_repeat_is_deterministic():
    wl = configs.ragged(seed=470, num_seqs=20)
    d = U.DeviceDecode(wl)
    d.append_all()
    a = d.attend().clone()
    b = d.attend().clone()
    assert torch.equal(a.view(torch.int32), b.view(torch.int32))


# ---------------------------------------------------------------------------
def test_bandwidth_config_full_size_all_sequences():
    """Batch 256 x context 2048 (1 GiB pool) in the automatic launch configuration the bench times;
    every sequence checked element by element against the oracle (one host thread per sequence)."""
    wl = configs.bandwidth()
    d = U.DeviceDecode(wl, fill_nan=False, generate_on_device=True)
    d.append_all()
    out = d.attend().cpu().double().numpy()
    assert d.status_value() == 0
    # the device generator reproduces the host stream bit for bit (checked on one sequence)
    from workloads import torch_gen
    kd, vd, _ = torch_gen.workload_kv(wl, 0, U.dev(), seqs=[77])
    kh, vh = wl.kv_tokens(77)
    assert np.array_equal(U.bits(kd), kh) and np.array_equal(U.bits(vd), vh)
    ref, err = U.oracle_decode_threaded(wl)
    assert err == 0
    U.assert_close(out, ref, "bandwidth, all 256 sequences")


# Equal-length batches in the automatic launch configuration (2 CTAs per SM, 304 on a
# 152-SM GB300) reach each branch of the kernel's split choice:
#  * n <= CTAs, each sequence cut into k > 1 equal parts and merged: 8 x 2048 (256 CTAs of
#    4 pages, 32 parts per sequence, merged in two levels) and 32 x 1024 (288 CTAs, 9 parts);
#  * n > CTAs with a divisor of n: whole sequences per CTA, 512 x 2048 (256 CTAs of 2
#    sequences, 2 GiB pool) and 608 x 512 (304 CTAs of 2);
#  * n > CTAs with no divisor in range (331 is prime): the even page split, every CTA's
#    range cutting sequences, 331 x 256.
@pytest.mark.parametrize("num_seqs,context", [(8, 2048), (32, 1024), (512, 2048), (608, 512), (331, 256)],
                         ids=["cut_8x2048", "cut_32x1024", "whole_512x2048", "whole_608x512", "prime_331x256"])
def test_equal_length_automatic_split_branches(num_seqs, context):
    wl = configs.custom(520 + num_seqs, [context] * num_seqs, name=f"equal_{num_seqs}x{context}")
    d = U.DeviceDecode(wl, fill_nan=True, generate_on_device=True)
    d.append_all()
    out = d.attend().cpu().double().numpy()
    assert d.status_value() == 0
    ref, err = U.oracle_decode_threaded(wl)
    assert err == 0
    U.assert_close(out, ref, wl.name)


def test_one_workspace_across_batch_sizes_and_splits():
    """The merge counters live at fixed slot positions and are reset by the merging CTA, so one
    zeroed workspace stays valid across calls with different batch sizes and CTA counts."""
    import paged_kv_cache_180_gb300 as pkv
    ws = pkv.decode_workspace(64, device=U.dev())
    for seed, n, ctas in ((480, 64, 0), (481, 5, 300), (482, 40, 17), (483, 64, 1024), (484, 3, 0)):
        wl = configs.ragged(seed=seed, num_seqs=n)
        d = U.DeviceDecode(wl)
        d.ws = ws
        d.append_all()
        out = d.attend(num_ctas=ctas).cpu().double().numpy()
        ref, err, _ = oracle.decode_workload(wl)
        U.assert_close(out, ref, f"batch {n}, ctas {ctas}")
        assert d.status_value() == 0
    # every completed call leaves both levels of merge counters at zero
    slot_bytes = 32 * 64 * 4 + 32 * 8 + 2 * 8 * 4
    counters = ws.view(-1, slot_bytes)[:, slot_bytes - 64:].contiguous().view(torch.int32)
    assert int(counters.abs().sum().item()) == 0


# ---------------------------------------------------------------------------
def _decode_step_case(wl, skip_every=0, layers=(0,)):
    """Pool holds every token but each sequence's last; one fused step appends it and attends."""
    import paged_kv_cache_180_gb300 as pkv
    from workloads import torch_gen
    d = U.DeviceDecode(wl)
    for layer in layers:
        k, v, slots = torch_gen.workload_kv(wl, layer, U.dev(), upto_offset=1)
        if slots.numel():
            pkv.kv_append(d.pool, k, v, slots, d.status)
    for layer in layers:
        kn, vn, sn = wl.decode_tokens(layer)
        sn = sn.copy()
        if skip_every:
            # these sequences' new tokens were appended earlier: slot -1 means "nothing to append"
            pre = np.arange(0, len(sn), skip_every)
            pkv.kv_append(d.pool, U.to_dev(kn[pre]), U.to_dev(vn[pre]), U.to_dev(sn[pre]), d.status)
            sn[pre] = -1
        blocks = wl.max_blocks
        pkv.decode_step(d.pool, U.to_dev(kn), U.to_dev(vn), U.to_dev(sn), d.out, d.q(layer),
                        d.bt.view(-1)[layer * blocks:], wl.num_layers * blocks, d.lens, wl.max_context, wl.scale,
                        d.ws, d.status)
        out = d.out.cpu().double().numpy()
        ref, err, opool = oracle.decode_workload(wl, layer=layer)
        assert err == 0
        U.assert_close(out, ref, f"decode_step {wl.name} layer {layer}")
    assert d.status_value() == 0
    # the pool now equals the oracle's after appending every token of every layer
    opool = oracle.Pool(wl.num_pages)
    for layer in layers:
        k, v, slots = wl.kv_all(layer)
        oracle.kv_append(opool, k, v, slots)
    np.testing.assert_array_equal(U.bits(d.pool.view()).reshape(-1), opool.data.reshape(-1))


def test_decode_step_fused_append_ragged():
    _decode_step_case(configs.ragged(seed=490, num_seqs=40))


def test_decode_step_with_skipped_appends_and_partial_pages():
    _decode_step_case(configs.custom(491, [1, 16, 17, 33, 2048, 300, 15, 32], name="fused_edges"), skip_every=3)


def test_decode_step_llama_layers():
    _decode_step_case(configs.llama_step(), layers=(0, 7, 15))


def test_decode_step_checks_the_new_tokens_slot():
    """The fused append stores a sequence's new token only at position ctx - 1 of its block
    table.  Another slot in the pool (an earlier row of the same page, another sequence's
    decode slot) or a slot past the pool sets PKV_DEV_BAD_SLOT, stores nothing and leaves the
    cached row in the softmax; a correct slot in the same call is stored and attended."""
    import paged_kv_cache_180_gb300 as pkv
    wl = configs.custom(497, [40, 16, 1, 300], name="slot_check")
    d = U.DeviceDecode(wl)
    d.append_all()                                    # every token cached, decode tokens included
    kn, vn, sn = wl.decode_tokens(0)
    r = np.random.default_rng(7)
    kn2 = rng.f64_to_bf16_bits(r.standard_normal(kn.shape))
    vn2 = rng.f64_to_bf16_bits(r.standard_normal(vn.shape))
    slots = sn.copy()
    slots[0] = sn[0] - 1                 # the row before the new token, same page
    slots[1] = sn[3]                     # sequence 3's decode slot
    slots[2] = wl.num_pages * 16 + 5     # past the pool
    blocks = wl.max_blocks
    pkv.decode_step(d.pool, U.to_dev(kn2), U.to_dev(vn2), U.to_dev(slots), d.out, d.q(0), d.bt.view(-1),
                    wl.num_layers * blocks, d.lens, wl.max_context, wl.scale, d.ws, d.status)
    assert d.status_value() == 1         # PKV_DEV_BAD_SLOT
    # expected: the cached pool, with only sequence 3's new token replaced
    _, err, opool = oracle.decode_workload(wl)
    assert err == 0
    assert oracle.kv_append(opool, kn2[3:4], vn2[3:4], sn[3:4]) == 0
    np.testing.assert_array_equal(U.bits(d.pool.view()).reshape(-1), opool.data.reshape(-1))
    bt = np.ascontiguousarray(wl.block_tables[:, 0, :])
    ref, err = oracle.paged_decode_attention(opool, wl.q(0), bt, wl.context_lens, wl.scale, wl.max_context)
    assert err == 0
    U.assert_close(d.out.cpu().double().numpy(), ref, "decode_step with checked slots")


@pytest.mark.parametrize("overlap", [False, True], ids=["serial", "overlap_previous"])
def test_graph_captured_llama_step_all_layers(overlap):
    """The 16-layer fused step (per-layer block-table slices) captured once as a CUDA graph
    and replayed twice: every layer's output matches the oracle and the replays leave the
    pool and the merge counters consistent.  With overlap_previous each layer's kernel may
    start (lengths, tables, first page copies) while the previous layer's finishes; the
    layers share the output buffer and the workspace, which are written only after the
    previous kernel completed."""
    import paged_kv_cache_180_gb300 as pkv
    from workloads import torch_gen
    wl = configs.llama_step()
    L, blocks = wl.num_layers, wl.max_blocks
    d = U.DeviceDecode(wl)
    for layer in range(L):
        k, v, slots = torch_gen.workload_kv(wl, layer, U.dev(), upto_offset=1)
        if slots.numel():
            pkv.kv_append(d.pool, k, v, slots, d.status)
    dec = [tuple(U.to_dev(a) for a in wl.decode_tokens(layer)) for layer in range(L)]
    qs = [d.q(layer) for layer in range(L)]
    outs = torch.empty((L, wl.num_seqs, 32, 64), dtype=torch.float32, device=U.dev())

    def step():
        for layer in range(L):
            kn, vn, sn = dec[layer]
            pkv.decode_step(d.pool, kn, vn, sn, outs[layer], qs[layer], d.bt.view(-1)[layer * blocks:], L * blocks,
                            d.lens, wl.max_context, wl.scale, d.ws, d.status, overlap_previous=overlap)

    step()
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        step()
    outs.fill_(float("nan"))
    g.replay()
    g.replay()
    torch.cuda.synchronize()
    assert d.status_value() == 0
    got = outs.cpu().double().numpy()
    for layer in range(L):
        ref, err, _ = oracle.decode_workload(wl, layer=layer)
        assert err == 0
        U.assert_close(got[layer], ref, f"graph replay, layer {layer}")


def test_decode_step_with_mapped_host_buffers():
    """q, the new K/V rows and the slots in pinned host memory (read by the kernel over the host
    link) and the output written straight to pinned host memory: same bits as the device run."""
    import paged_kv_cache_180_gb300 as pkv
    from workloads import torch_gen
    wl = configs.ragged(seed=492, num_seqs=24)
    outs = []
    for mapped in (False, True):
        d = U.DeviceDecode(wl)
        k, v, slots = torch_gen.workload_kv(wl, 0, U.dev(), upto_offset=1)
        if slots.numel():
            pkv.kv_append(d.pool, k, v, slots, d.status)
        kn, vn, sn = (U.to_dev(a) for a in wl.decode_tokens(0))
        q = d.q(0)
        out = d.out
        if mapped:
            kn, vn, sn, q = (x.cpu().pin_memory() for x in (kn, vn, sn, q))
            out = torch.full(tuple(d.out.shape), float("nan"), dtype=torch.float32).pin_memory()
        pkv.decode_step(d.pool, kn, vn, sn, out, q, d.bt.view(-1), wl.num_layers * wl.max_blocks, d.lens,
                        wl.max_context, wl.scale, d.ws, d.status)
        assert d.status_value() == 0
        outs.append(out.cpu().clone())
        if mapped:
            ref, err, opool = oracle.decode_workload(wl, layer=0)
            assert err == 0
            U.assert_close(outs[-1].double().numpy(), ref, "decode_step, mapped host buffers")
            np.testing.assert_array_equal(U.bits(d.pool.view()).reshape(-1), opool.data.reshape(-1))
    assert torch.equal(outs[0], outs[1])


def test_kv_append_from_mapped_host_buffers():
    import paged_kv_cache_180_gb300 as pkv
    wl = configs.ragged(seed=493, num_seqs=8)
    d = U.DeviceDecode(wl)
    k, v, slots = wl.kv_all(0)
    kh, vh, sh = (U.to_dev(a).cpu().pin_memory() for a in (k, v, slots))
    pkv.kv_append(d.pool, kh, vh, sh, d.status)
    assert d.status_value() == 0
    opool = oracle.Pool(wl.num_pages)
    oracle.kv_append(opool, k, v, slots)
    np.testing.assert_array_equal(U.bits(d.pool.view()).reshape(-1), opool.data.reshape(-1))


def test_overlapped_steps_sharing_output_and_workspace():
    """Eager launches with overlap_previous: 16 layers written to ONE output buffer and one
    workspace, each layer's kernel allowed to start during the previous one's; the buffer
    ends with the last layer's result, and every layer checked on its own run matches."""
    import paged_kv_cache_180_gb300 as pkv
    from workloads import torch_gen
    wl = configs.llama_step()
    L, blocks = wl.num_layers, wl.max_blocks
    d = U.DeviceDecode(wl)
    for layer in range(L):
        k, v, slots = torch_gen.workload_kv(wl, layer, U.dev(), upto_offset=1)
        if slots.numel():
            pkv.kv_append(d.pool, k, v, slots, d.status)
    dec = [tuple(U.to_dev(a) for a in wl.decode_tokens(layer)) for layer in range(L)]
    qs = [d.q(layer) for layer in range(L)]
    copies = []
    for layer in range(L):
        kn, vn, sn = dec[layer]
        pkv.decode_step(d.pool, kn, vn, sn, d.out, qs[layer], d.bt.view(-1)[layer * blocks:], L * blocks, d.lens,
                        wl.max_context, wl.scale, d.ws, d.status, overlap_previous=True)
        copies.append(d.out.clone())  # a copy kernel between the steps: ordinary stream order
    assert d.status_value() == 0
    for layer in (0, 5, 15):
        ref, err, _ = oracle.decode_workload(wl, layer=layer)
        assert err == 0
        U.assert_close(copies[layer].cpu().double().numpy(), ref, f"overlapped eager, layer {layer}")
    # back to back with no copy in between: the shared output holds the last layer
    for layer in range(L):
        kn, vn, sn = dec[layer]
        pkv.decode_step(d.pool, kn, vn, sn, d.out, qs[layer], d.bt.view(-1)[layer * blocks:], L * blocks, d.lens,
                        wl.max_context, wl.scale, d.ws, d.status, overlap_previous=True)
    assert d.status_value() == 0
    assert torch.equal(d.out, copies[L - 1])


def test_overlapped_step_reads_q_written_by_the_kernel_before():
    """A small batch (the clustered instance, which starts its query lines toward L2 before it
    waits for the kernel before it) launched with overlap_previous right after a kv_append
    that writes the very bytes it then reads as q: the K half of a spare page, 16 appended
    tokens of 8 heads, is the 4 x 32 x 64 query block.  The outputs must match the oracle fed
    with the bytes of its own append, on every repetition (new values each time)."""
    import paged_kv_cache_180_gb300 as pkv
    from workloads import torch_gen
    lens = [128, 512, 1024, 2048]
    need = sum(-(-c // 16) for c in lens)
    wl = configs.custom(191, lens, num_pages=need + 64, name="q-written-before")
    used = set(int(x) for x in wl.block_tables[:, 0, :].reshape(-1) if x >= 0)
    spare = [pg for pg in range(wl.num_pages) if pg not in used]
    assert len(spare) == 64
    qpage = spare[0]
    d = U.DeviceDecode(wl)
    k, v, slots = torch_gen.workload_kv(wl, 0, U.dev(), upto_offset=1)
    pkv.kv_append(d.pool, k, v, slots, d.status)
    kn, vn, sn = (U.to_dev(a) for a in wl.decode_tokens(0))
    q_dev = d.pool.view()[qpage, 0].view(4, 32, 64)  # the spare page's K half itself, read as q
    _, err, opool = oracle.decode_workload(wl)
    assert err == 0
    spare_slots = np.array([pg * 16 + r for pg in spare for r in range(16)], dtype=np.int32)
    n = spare_slots.size * 8 * 64
    bt0 = np.ascontiguousarray(wl.block_tables[:, 0, :])
    for rep in range(6):
        ks = rng.normal_bf16(rng.stream_key(191, f"spare-k-{rep}"), 0, n).reshape(-1, 8, 64)
        vs = rng.normal_bf16(rng.stream_key(191, f"spare-v-{rep}"), 0, n).reshape(-1, 8, 64)
        pkv.kv_append(d.pool, U.to_dev(ks), U.to_dev(vs), U.to_dev(spare_slots), d.status)
        pkv.decode_step(d.pool, kn, vn, sn, d.out, q_dev, d.bt.view(-1), wl.max_blocks, d.lens, wl.max_context,
                        wl.scale, d.ws, d.status, overlap_previous=True)
        assert d.status_value() == 0
        assert oracle.kv_append(opool, ks, vs, spare_slots) == 0
        q_host = np.ascontiguousarray(opool.data[qpage, 0]).reshape(4, 32, 64)
        ref, err = oracle.paged_decode_attention(opool, q_host, bt0, wl.context_lens, wl.scale, wl.max_context)
        assert err == 0
        U.assert_close(d.out.cpu().double().numpy(), ref, f"q written by the append before, repetition {rep}")


@pytest.mark.parametrize("pad", [0, 256], ids=["packed", "padded_stride"])
def test_separate_k_and_v_buffers(pad):
    """K and V pools in two separate allocations with a page stride of half a page (plus
    optional padding): append bit-exact per half, decode and prefill match the oracle."""
    import paged_kv_cache_180_gb300 as pkv
    wl = configs.ragged(seed=494, num_seqs=12)
    half_elems = 8 * 16 * 64
    stride = half_elems * 2 + pad                       # bytes between pages
    n_elems = (wl.num_pages * stride) // 2
    kbuf = torch.full((n_elems,), -1, dtype=torch.int16, device=U.dev()).view(torch.bfloat16)
    vbuf = torch.full((n_elems,), -1, dtype=torch.int16, device=U.dev()).view(torch.bfloat16)
    desc = pkv.kv_pool_create(kbuf, vbuf, stride, wl.num_pages)
    status = torch.zeros(1, dtype=torch.int32, device=U.dev())
    k, v, slots = wl.kv_all(0)
    pkv.kv_append(desc, U.to_dev(k), U.to_dev(v), U.to_dev(slots), status)
    opool = oracle.Pool(wl.num_pages)
    oracle.kv_append(opool, k, v, slots)
    for buf, ref_half in ((kbuf, opool.k), (vbuf, opool.v)):
        pages = U.bits(buf).reshape(wl.num_pages, stride // 2)[:, :half_elems].reshape(ref_half.shape)
        np.testing.assert_array_equal(pages, ref_half)
    # decode
    out = torch.empty(wl.num_seqs, 32, 64, dtype=torch.float32, device=U.dev())
    ws = pkv.decode_workspace(wl.num_seqs, device=U.dev())
    bt_host = np.ascontiguousarray(wl.block_tables[:, 0, :])
    bt, lens = U.to_dev(bt_host), U.to_dev(wl.context_lens)
    pkv.paged_decode_attention(desc, out, U.to_dev(wl.q(0)), bt, bt_host.shape[1], lens, wl.max_context, wl.scale,
                               ws, status)
    assert int(status.item()) == 0
    ref, err, _ = oracle.decode_workload(wl)
    assert err == 0
    U.assert_close(out.cpu().double().numpy(), ref, "decode, separate K and V buffers")
    # prefill of the last min(ctx, 24) tokens
    nq = [min(int(c), 24) for c in wl.context_lens]
    qs = np.concatenate([[0], np.cumsum(nq)]).astype(np.int32)
    total = int(qs[-1])
    qbits = rng.normal_bf16(rng.stream_key(494, "pf-q"), 0, total * 32 * 64).reshape(total, 32, 64)
    pout = torch.full((total, 32, 64), float("nan"), dtype=torch.float32, device=U.dev())
    pkv.paged_prefill_attention(desc, pout, U.to_dev(qbits), U.to_dev(qs), bt, bt_host.shape[1], lens, max(nq),
                                wl.max_context, wl.scale, status)
    assert int(status.item()) == 0
    pref, perr = oracle.paged_prefill_attention(opool, qbits, qs, bt_host, wl.context_lens, wl.scale, wl.max_context)
    assert perr == 0
    U.assert_close(pout.cpu().double().numpy(), pref, "prefill, separate K and V buffers")


def test_calls_run_on_the_callers_stream():
    """Append and attention enqueued on a side stream (as the current stream, and passed
    explicitly) are ordered on that stream and match the oracle."""
    import paged_kv_cache_180_gb300 as pkv
    wl = configs.ragged(seed=495, num_seqs=10)
    side = torch.cuda.Stream()
    d = U.DeviceDecode(wl)
    k, v, slots = (U.to_dev(a) for a in wl.kv_all(0))
    q = d.q(0)
    torch.cuda.synchronize()
    with torch.cuda.stream(side):
        pkv.kv_append(d.pool, k, v, slots, d.status)  # on the current (side) stream
    blocks = wl.max_blocks
    pkv.paged_decode_attention(d.pool, d.out, q, d.bt.view(-1), wl.num_layers * blocks, d.lens, wl.max_context,
                               wl.scale, d.ws, d.status, stream=side)  # passed explicitly
    side.synchronize()
    assert int(d.status.item()) == 0
    ref, err, _ = oracle.decode_workload(wl)
    assert err == 0
    U.assert_close(d.out.cpu().double().numpy(), ref, "side stream")


def test_status_word_is_optional():
    """device_status may be null: calls with no status word (a valid batch, and one with an
    invalid context that would set a bit) run and give the same rows."""
    import paged_kv_cache_180_gb300 as pkv
    wl = configs.ragged(seed=496, num_seqs=6)
    d = U.DeviceDecode(wl)
    d.append_all()
    blocks = wl.max_blocks
    q = d.q(0)
    pkv.paged_decode_attention(d.pool, d.out, q, d.bt.view(-1), wl.num_layers * blocks, d.lens, wl.max_context,
                               wl.scale, d.ws, None)
    torch.cuda.synchronize()
    ref, err, _ = oracle.decode_workload(wl)
    assert err == 0
    U.assert_close(d.out.cpu().double().numpy(), ref, "no status word")
    bad_lens = d.lens.clone()
    bad_lens[2] = wl.max_context + 1
    pkv.paged_decode_attention(d.pool, d.out, q, d.bt.view(-1), wl.num_layers * blocks, bad_lens, wl.max_context,
                               wl.scale, d.ws, None)
    torch.cuda.synchronize()
    got = d.out.cpu().double().numpy()
    assert np.isfinite(got).all() and not got[2].any()   # the invalid sequence's rows are zeros
    keep = [s for s in range(wl.num_seqs) if s != 2]
    U.assert_close(got[keep], ref[keep], "no status word, one invalid context")
