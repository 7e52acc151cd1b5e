"""Pins for the oracle's paged prefill attention (no GPU).

* torch.nn.functional.scaled_dot_product_attention in float64 on logical (never
  paged) K/V with an explicit boolean mask "key t <= position of the query" - a
  library routine, and a different formulation from the oracle's per-row loop;
* with one query per sequence it is the decode oracle (position = ctx - 1);
* the first query of a fresh prefill sees only token 0: its output is V[0] exactly;
* causality: changing the K/V of tokens after a query's position leaves that query's
  output bit-identical and changes the later queries';
* error bits for more queries than context;
* planted mistakes (mask off by one, wrong position base) are caught.
"""
import math
import os
import subprocess
import sys
import tempfile

import numpy as np
import pytest
import torch

import oracle
from tests.test_oracle import as_f64, build_case
from workloads import rng

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def torch_prefill(q_bits, k_bits, v_bits, n, scale):
    """SDPA over the first ctx tokens for the last n query positions, float64."""
    q = torch.from_numpy(as_f64(q_bits)).permute(1, 0, 2)        # [Hq, n, D]
    k = torch.from_numpy(as_f64(k_bits))                          # [ctx, Hkv, D]
    v = torch.from_numpy(as_f64(v_bits))
    ctx = k.shape[0]
    group = q.shape[0] // k.shape[1]
    k = torch.repeat_interleave(k, group, dim=1).permute(1, 0, 2)  # [Hq, ctx, D]
    v = torch.repeat_interleave(v, group, dim=1).permute(1, 0, 2)
    pos = torch.arange(ctx - n, ctx)[:, None]
    mask = torch.arange(ctx)[None, :] <= pos                      # [n, ctx]
    o = torch.nn.functional.scaled_dot_product_attention(q, k, v, attn_mask=mask, scale=scale)
    return o.permute(1, 0, 2).numpy()                             # [n, Hq, D]


def prefill_case(seed, lens, nq, num_q_heads=32, num_kv_heads=8, head_dim=64, page_tokens=16):
    c = build_case(seed, lens, num_q_heads, num_kv_heads, head_dim, page_tokens)
    qs = np.concatenate([[0], np.cumsum(nq)]).astype(np.int32)
    qkey = rng.stream_key(seed, "prefill-q")
    total = int(qs[-1])
    q = rng.normal_bf16(qkey, 0, total * num_q_heads * head_dim).reshape(total, num_q_heads, head_dim)
    c.update(qs=qs, qp=q, nq=list(nq))
    return c


def run_oracle(c, scale=0.125):
    return oracle.paged_prefill_attention(c["pool"], c["qp"], c["qs"], c["bt"], c["lens"], scale, c["max_context"])


@pytest.mark.parametrize("case", range(40))
def test_prefill_vs_torch_sdpa(case):
    r = np.random.default_rng(300 + case)
    page_tokens = int(r.choice([2, 4, 16]))
    num_kv_heads = int(r.integers(1, 4))
    group = int(r.integers(1, 5))
    head_dim = int(r.choice([8, 16, 64]))
    nseq = int(r.integers(1, 4))
    lens = r.integers(1, 50, size=nseq)
    nq = [int(r.integers(1, int(c_) + 1)) for c_ in lens]
    c = prefill_case(700 + case, lens, nq, group * num_kv_heads, num_kv_heads, head_dim, page_tokens)
    out, err = run_oracle(c)
    assert err == 0
    for s in range(nseq):
        a, b = c["qs"][s], c["qs"][s + 1]
        ref = torch_prefill(c["qp"][a:b], c["k"][s], c["v"][s], nq[s], 0.125)
        np.testing.assert_allclose(out[a:b], ref, rtol=1e-12, atol=1e-13)


def test_single_query_is_decode():
    c = prefill_case(31, [37, 16, 5], [1, 1, 1])
    out, err = run_oracle(c)
    dec, err2 = oracle.paged_decode_attention(c["pool"], c["qp"], c["bt"], c["lens"], 0.125, c["max_context"])
    assert err == err2 == 0
    assert np.array_equal(out, dec)


def test_first_query_of_fresh_prefill_is_v0():
    c = prefill_case(32, [23, 9], [23, 9])
    out, err = run_oracle(c)
    assert err == 0
    for s in range(2):
        v0 = np.repeat(as_f64(c["v"][s][0]), 4, axis=0)
        assert np.array_equal(out[c["qs"][s]], v0)


def test_causality():
    lens, nq = [40], [12]
    c = prefill_case(33, lens, nq)
    out1, _ = run_oracle(c)
    # overwrite K/V of tokens 35.. (positions after query j = 35 - 28 = 7)
    cut = 35
    t = np.arange(cut, 40)
    slots = (c["bt"][0, t // 16].astype(np.int64) * 16 + t % 16).astype(np.int32)
    junk = rng.f64_to_bf16_bits(np.random.default_rng(5).standard_normal((len(t), 8, 64)) * 3)
    oracle.kv_append(c["pool"], junk, junk, slots)
    out2, _ = run_oracle(c)
    first_query = 40 - 12
    for j in range(12):
        pos = first_query + j
        if pos < cut:
            assert np.array_equal(out1[j], out2[j]), j
        else:
            assert not np.allclose(out1[j], out2[j]), j


def test_error_bits():
    c = prefill_case(34, [10, 20], [11, 5])
    out, err = run_oracle(c)
    assert err == oracle.ERR_CONTEXT
    assert not out[:11].any() and out[11:].any()


MUTANTS = {
    "mask_off_by_one": ("pos + 1, scale,\n                                x)", "pos, scale,\n                                x)"),
    "position_base": ("int pos = ctx - n + j;", "int pos = ctx - n + j - (j > 0);"),
    "gqa": ("            int g = h / group;\n                const uint16_t *qh = q + ((int64_t)(q0 + j)",
            "            int g = h % num_kv_heads;\n                const uint16_t *qh = q + ((int64_t)(q0 + j)"),
}


@pytest.mark.parametrize("name", sorted(MUTANTS))
def test_planted_prefill_mistake_is_caught(name):
    old, new = MUTANTS[name]
    src = open(os.path.join(ROOT, "oracle", "pkv_oracle.c")).read()
    assert src.count(old) == 1, name
    with tempfile.TemporaryDirectory() as d:
        path = os.path.join(d, "m.c")
        open(path, "w").write(src.replace(old, new))
        so = os.path.join(d, "libm.so")
        subprocess.check_call(["gcc", "-std=c99", "-O2", "-ffp-contract=off", "-shared", "-fPIC", "-o", so, path,
                               "-lm"])
        code = ("import sys; sys.path.insert(0, %r); import oracle; oracle.use_library(%r)\n"
                "from tests import test_oracle_prefill as t\n"
                "caught = []\n"
                "for f in (lambda: t.test_prefill_vs_torch_sdpa(3), lambda: t.test_prefill_vs_torch_sdpa(11),"
                " t.test_first_query_of_fresh_prefill_is_v0, t.test_causality):\n"
                "    try: f()\n"
                "    except AssertionError: caught.append(1)\n"
                "print('CAUGHT' if caught else 'MISSED')\n") % (ROOT, so)
        r = subprocess.run([sys.executable, "-c", code], capture_output=True, text=True, cwd=ROOT, timeout=300)
        assert r.returncode < 0 or "CAUGHT" in r.stdout, r.stdout + r.stderr
