"""Pins for the CPU oracle (no GPU).

The oracle is checked against things other than itself:
  * a hand-derived worked example of the pool layout (tests/golden/append_layout.txt);
  * a second, independent formulation: the logical (never paged) K/V, heads
    expanded with torch.repeat_interleave and weights from torch.softmax in
    float64 - a library routine and a different formula (x - logsumexp);
  * closed forms and invariants: one-token context returns V exactly, equal keys
    and q = 0 return the mean of V, weights sum to one, weight ratios equal
    exp(scale * score difference) for integer-valued dot products, a dominant
    score returns its V row, query head h reads K/V head h // group, physical
    page order does not change the result;
  * the error bits for bad slots, bad context lengths and unassigned pages.
"""
import math
import os

import numpy as np
import pytest
import torch

import oracle
from workloads import configs, rng

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def bf16(x) -> np.ndarray:
    return rng.f64_to_bf16_bits(np.asarray(x, dtype=np.float64))


def as_f64(bits) -> np.ndarray:
    return rng.bf16_bits_to_f64(bits)


def build_case(seed, lens, num_q_heads=32, num_kv_heads=8, head_dim=64, page_tokens=16, extra_pages=3,
               max_blocks=None):
    """Random paged case: logical K/V/q plus a pool filled through the oracle's append."""
    lens = np.asarray(lens, dtype=np.int32)
    blocks = [math.ceil(int(c) / page_tokens) for c in lens]
    max_blocks = max_blocks or max(max(blocks), 1)
    num_pages = sum(blocks) + extra_pages
    perm = list(rng.permutation(rng.stream_key(seed, "perm"), num_pages))
    bt = np.full((len(lens), max_blocks), -1, dtype=np.int32)
    for s, nb in enumerate(blocks):
        for j in range(nb):
            bt[s, j] = perm.pop()
    kkey, vkey, qkey = (rng.stream_key(seed, t) for t in ("k", "v", "q"))
    te = num_kv_heads * head_dim
    ks, vs = [], []
    pool = oracle.Pool(num_pages, page_tokens, num_kv_heads, head_dim)
    off = 0
    for s, c in enumerate(lens):
        c = int(c)
        k = rng.normal_bf16(kkey, off, c * te).reshape(c, num_kv_heads, head_dim)
        v = rng.normal_bf16(vkey, off, c * te).reshape(c, num_kv_heads, head_dim)
        off += c * te
        t = np.arange(c)
        slots = (bt[s, t // page_tokens].astype(np.int64) * page_tokens + t % page_tokens).astype(np.int32)
        assert oracle.kv_append(pool, k, v, slots) == 0
        ks.append(k)
        vs.append(v)
    q = rng.normal_bf16(qkey, 0, len(lens) * num_q_heads * head_dim).reshape(len(lens), num_q_heads, head_dim)
    return dict(pool=pool, bt=bt, lens=lens, q=q, k=ks, v=vs, max_context=max_blocks * page_tokens)


def torch_reference(q_bits, k_bits, v_bits, scale):
    """softmax(scale * q K^T) V on logical (contiguous) K/V, float64, via torch library routines."""
    q = torch.from_numpy(as_f64(q_bits))                       # [Hq, D]
    k = torch.from_numpy(as_f64(k_bits))                       # [T, Hkv, D]
    v = torch.from_numpy(as_f64(v_bits))
    group = q.shape[0] // k.shape[1]
    k = torch.repeat_interleave(k, group, dim=1)               # [T, Hq, D]
    v = torch.repeat_interleave(v, group, dim=1)
    scores = torch.einsum("hd,thd->ht", q, k) * scale
    w = torch.softmax(scores, dim=-1)
    return torch.einsum("ht,thd->hd", w, v).numpy()


# ---------------------------------------------------------------------------
def test_append_layout_golden():
    lines = [ln.split("#")[0].strip() for ln in open(os.path.join(GOLDEN, "append_layout.txt"))]
    lines = [ln for ln in lines if ln]
    geo = dict(kv.split("=") for kv in lines[0].split()[1:])
    pt, hk, hd, npg, fill = (int(geo[k]) for k in ("page_tokens", "num_kv_heads", "head_dim", "num_pages", "fill"))
    appends = [tuple(map(int, ln.split()[1:])) for ln in lines if ln.startswith("append")]
    expect = dict(tuple(map(int, ln.split())) for ln in lines[1:] if not ln.startswith("append"))
    n = len(appends)
    k_new = np.zeros((n, hk, hd), np.uint16)
    v_new = np.zeros((n, hk, hd), np.uint16)
    for i, _ in appends:
        for g in range(hk):
            for d in range(hd):
                k_new[i, g, d] = 100 * (i + 1) + 10 * g + d
                v_new[i, g, d] = 100 * (i + 1) + 10 * g + d + 50
    slots = np.array([s for _, s in appends], np.int32)
    pool = oracle.Pool(npg, pt, hk, hd, fill=fill)
    assert oracle.kv_append(pool, k_new, v_new, slots) == 0
    flat = pool.data.reshape(-1)
    want = np.full(flat.shape, fill, np.uint16)
    for idx, val in expect.items():
        want[idx] = val
    np.testing.assert_array_equal(flat, want)


def test_append_bad_slot_reported_and_skipped():
    pool = oracle.Pool(2, 4, 1, 2)
    before = pool.data.copy()
    k = np.ones((1, 1, 2), np.uint16)
    assert oracle.kv_append(pool, k, k, np.array([8], np.int32)) == oracle.ERR_SLOT
    np.testing.assert_array_equal(pool.data, before)


def test_tiny_config_vs_torch():
    wl = configs.tiny()
    out, err, _ = oracle.decode_workload(wl)
    assert err == 0
    k, v = wl.kv_tokens(0)
    ref = torch_reference(wl.q()[0], k, v, wl.scale)
    np.testing.assert_allclose(out[0], ref, rtol=1e-12, atol=1e-13)


@pytest.mark.parametrize("case", range(200))
def test_random_tiny_vs_torch(case):
    r = np.random.default_rng(1000 + case)
    page_tokens = int(r.choice([1, 2, 4, 8, 16]))
    num_kv_heads = int(r.integers(1, 5))
    group = int(r.integers(1, 5))
    head_dim = int(r.choice([4, 8, 16, 64]))
    nseq = int(r.integers(1, 4))
    lens = r.integers(1, 41, size=nseq)
    lens = np.minimum(lens, 8 * page_tokens)
    c = build_case(5000 + case, lens, group * num_kv_heads, num_kv_heads, head_dim, page_tokens)
    out, err = oracle.paged_decode_attention(c["pool"], c["q"], c["bt"], c["lens"], 0.125, c["max_context"])
    assert err == 0
    for s in range(nseq):
        ref = torch_reference(c["q"][s], c["k"][s], c["v"][s], 0.125)
        np.testing.assert_allclose(out[s], ref, rtol=1e-12, atol=1e-13)


def test_page_permutation_invariance_bit_exact():
    c = build_case(7, [37, 16, 1, 50], extra_pages=5)
    out1, e1 = oracle.paged_decode_attention(c["pool"], c["q"], c["bt"], c["lens"], 0.125, c["max_context"])
    # Move every page to a new physical id and rewrite the tables accordingly.
    n = c["pool"].num_pages
    perm = rng.permutation(rng.stream_key(99, "move"), n)   # old id -> new id
    pool2 = oracle.Pool(n, 16, 8, 64)
    pool2.data[perm] = c["pool"].data
    bt2 = np.where(c["bt"] >= 0, perm[np.maximum(c["bt"], 0)], -1).astype(np.int32)
    out2, e2 = oracle.paged_decode_attention(pool2, c["q"], bt2, c["lens"], 0.125, c["max_context"])
    assert e1 == e2 == 0
    assert np.array_equal(out1, out2)


def test_one_token_context_returns_v_exactly():
    c = build_case(8, [1, 1])
    out, err = oracle.paged_decode_attention(c["pool"], c["q"], c["bt"], c["lens"], 0.125, c["max_context"])
    assert err == 0
    for s in range(2):
        v = as_f64(c["v"][s][0])                      # [Hkv, D]
        want = np.repeat(v, 4, axis=0)                # query head h reads kv head h // 4
        assert np.array_equal(out[s], want)


def _case_with(k_vals, v_vals, q_vals, page_tokens=16, seed=3):
    """Single sequence with explicit K/V/q values (float arrays, rounded to bf16)."""
    ctx = k_vals.shape[0]
    c = build_case(seed, [ctx], q_vals.shape[0], k_vals.shape[1], k_vals.shape[2], page_tokens)
    pool = oracle.Pool(c["pool"].num_pages, page_tokens, k_vals.shape[1], k_vals.shape[2])
    t = np.arange(ctx)
    slots = (c["bt"][0, t // page_tokens].astype(np.int64) * page_tokens + t % page_tokens).astype(np.int32)
    kb, vb = bf16(k_vals), bf16(v_vals)
    assert oracle.kv_append(pool, kb, vb, slots) == 0
    qb = bf16(q_vals)[None]
    return pool, c["bt"], np.array([ctx], np.int32), qb, c["max_context"], kb, vb


def test_identical_keys_and_zero_query_give_mean_of_v():
    r = np.random.default_rng(11)
    ctx = 45
    v = r.standard_normal((ctx, 8, 64))
    key = r.standard_normal((1, 8, 64))
    k_same = np.repeat(key, ctx, axis=0)
    q = r.standard_normal((32, 64))
    for k_vals, q_vals in ((k_same, q), (r.standard_normal((ctx, 8, 64)), np.zeros((32, 64)))):
        pool, bt, lens, qb, mc, _, vb = _case_with(k_vals, v, q_vals)
        out, err = oracle.paged_decode_attention(pool, qb, bt, lens, 0.125, mc)
        assert err == 0
        mean_v = np.repeat(as_f64(vb).mean(axis=0), 4, axis=0)
        np.testing.assert_allclose(out[0], mean_v, rtol=1e-12, atol=1e-12)


def test_weights_sum_to_one_and_ratio_closed_form():
    # Integer-valued q and K make every dot product an exact integer, so the
    # weight ratio w_i / w_j must equal exp(scale * (dot_i - dot_j)).
    r = np.random.default_rng(12)
    ctx = 33
    k = r.integers(-3, 4, size=(ctx, 8, 64)).astype(np.float64)
    v = r.standard_normal((ctx, 8, 64))
    q = r.integers(-2, 3, size=(32, 64)).astype(np.float64)
    pool, bt, lens, qb, _, _, _ = _case_with(k, v, q)
    for h in (0, 5, 31):
        w, err = oracle.attention_weights(pool, qb, bt, lens, 0, h, 0.125)
        assert err == 0
        assert abs(w.sum() - 1.0) <= 1e-12
        dots = k[:, h // 4, :] @ q[h]
        for i, j in ((0, 1), (5, 17), (32, 3)):
            assert math.isclose(w[i] / w[j], math.exp(0.125 * (dots[i] - dots[j])), rel_tol=1e-12)


@pytest.mark.parametrize("row", [
    # score-row stress shapes (values chosen here): ordinary, tied maximum,
    # one dominant score, all negative, a full 16-token page
    [0.5, 1.5, -2.0, 3.0, 0.25, 2.0, -0.75, 1.0],
    [2.5] * 8,
    [0.0078125] * 3 + [40.0] + [0.0078125] * 4,
    [0.5] * 5 + [2048.0] + [0.5] * 2,
    [-6.0, -2.0, -9.0, -0.5, -7.0, -3.0, -4.0, -1.5],
    [0.5, -1.0, 2.0, 3.5, -2.5, 4.0, 1.0, 0.0, -3.0, 6.0, 2.5, -0.25, 1.5, -5.0, 3.0, 0.75],
])
def test_score_row_shapes(row):
    # q = 8 * e_0 and K[t][0] = score_t, so with scale 1/8 the score of token t is exactly row[t].
    n = len(row)
    k = np.zeros((n, 8, 64))
    k[:, :, 0] = np.asarray(row)[:, None]
    q = np.zeros((32, 64))
    q[:, 0] = 8.0
    v = np.random.default_rng(13).standard_normal((n, 8, 64))
    pool, bt, lens, qb, _, _, _ = _case_with(k, v, q)
    w, err = oracle.attention_weights(pool, qb, bt, lens, 0, 0, 0.125)
    assert err == 0
    assert np.all(np.isfinite(w)) and np.all(w >= 0)
    assert abs(w.sum() - 1.0) <= 1e-12
    top = int(np.argmax(row))
    for t in range(n):
        assert math.isclose(w[t] / w[top], math.exp(row[t] - row[top]), rel_tol=1e-12, abs_tol=1e-300)
    if len(set(row)) == 1:
        np.testing.assert_allclose(w, np.full(n, 1.0 / n), rtol=1e-15)


def test_dominant_score_selects_its_row_and_token_order():
    # V of token t is the constant t; a query aligned with one key picks that
    # token, which pins the page/row indexing of every token in the context.
    ctx = 70
    for j in (0, 15, 16, 31, 47, 69):
        k = np.zeros((ctx, 8, 64))
        k[j, :, 1] = 64.0
        v = np.broadcast_to(np.arange(ctx, dtype=np.float64)[:, None, None], (ctx, 8, 64)).copy()
        q = np.zeros((32, 64))
        q[:, 1] = 64.0
        pool, bt, lens, qb, mc, _, _ = _case_with(k, v, q, seed=20 + j)
        out, err = oracle.paged_decode_attention(pool, qb, bt, lens, 0.125, mc)
        assert err == 0
        # score_j = 0.125 * 64 * 64 = 512, others 0: weight of the rest ~ ctx * e^-512
        np.testing.assert_allclose(out[0], np.full((32, 64), float(j)), rtol=0, atol=1e-200)


def test_gqa_head_mapping():
    # V of kv head g is the constant g; every query head h must read g = h // group.
    ctx = 20
    for num_kv, group in ((8, 4), (2, 3), (4, 1)):
        r = np.random.default_rng(num_kv * 10 + group)
        k = r.standard_normal((ctx, num_kv, 16))
        v = np.broadcast_to(np.arange(num_kv, dtype=np.float64)[None, :, None], (ctx, num_kv, 16)).copy()
        q = r.standard_normal((num_kv * group, 16))
        pool, bt, lens, qb, mc, _, _ = _case_with(k, v, q, page_tokens=4)
        out, err = oracle.paged_decode_attention(pool, qb, bt, lens, 0.125, mc)
        assert err == 0
        want = (np.arange(num_kv * group) // group).astype(np.float64)
        np.testing.assert_allclose(out[0], np.broadcast_to(want[:, None], out[0].shape), rtol=0, atol=1e-14)


def test_context_zero_and_error_bits():
    c = build_case(9, [5, 20, 3])
    lens = c["lens"].copy()
    lens[0] = 0
    out, err = oracle.paged_decode_attention(c["pool"], c["q"], c["bt"], lens, 0.125, c["max_context"])
    assert err == 0 and not out[0].any() and out[1].any()
    lens[2] = c["max_context"] + 1
    out, err = oracle.paged_decode_attention(c["pool"], c["q"], c["bt"], lens, 0.125, c["max_context"])
    assert err == oracle.ERR_CONTEXT and not out[2].any()
    bt = c["bt"].copy()
    bt[1, 1] = -1
    out, err = oracle.paged_decode_attention(c["pool"], c["q"], bt, c["lens"], 0.125, c["max_context"])
    assert err == oracle.ERR_PAGE and not out[1].any() and out[0].any()
    bt[1, 1] = c["pool"].num_pages
    out, err = oracle.paged_decode_attention(c["pool"], c["q"], bt, c["lens"], 0.125, c["max_context"])
    assert err == oracle.ERR_PAGE


def test_llama_step_layer_sample_vs_torch():
    # One sequence of the 16-layer config (context 512, with the x8 K spikes), one layer.
    wl = configs.llama_step()
    out, err, _ = oracle.decode_workload(wl, layer=5, seqs=[1])
    assert err == 0
    k, v = wl.kv_tokens(1, 5)
    ref = torch_reference(wl.q(5)[1], k, v, wl.scale)
    np.testing.assert_allclose(out[1], ref, rtol=1e-11, atol=1e-12)
    assert not out[0].any()
